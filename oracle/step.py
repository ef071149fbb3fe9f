"""Float64 statement of each part of the structured-read denoise step.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function takes
plain NumPy arrays already rounded to the storage precision the GPU path reads
(bf16 values held in float32, fp32 temperatures) and computes in float64 with
dense matrices and explicit masks: no streaming, no tiling, no fusion.

Readings of points the pages leave open are listed next to the code that
takes them; each is also listed in the design notes of the repository.
"""
import numpy as np

from .philox import noise_tokens

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------
def bf16_round(x):
    """Round float32 values to the nearest bfloat16 (ties to even), as float32.

    The GPU forms a noised slot row and the next-step hidden row as an fp32
    sum rounded to bf16 because its GEMMs take bf16 operands; the oracle makes
    the same rounding so that both sides feed the same operand.
    """
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    out = u.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), x, out)


# --------------------------------------------------------------------------
# a1: decoder-mode attention
# --------------------------------------------------------------------------
def paged_to_contiguous(pool_k, pool_v, page_table, prompt_len, page_size):
    """Gather a paged encoder KV cache into per-request contiguous arrays.

    pool_k/pool_v: [n_pages, page_size, Hkv, d]; page_table: [B, max_pages]
    (page index of each page_size-token block of request b's prompt);
    key j of request b sits at pool[page_table[b, j // page_size], j % page_size].
    Returns kenc, venc of shape [B, max(prompt_len), Hkv, d] (zero past the end).
    """
    B = page_table.shape[0]
    pmax = int(max(prompt_len)) if B else 0
    _, _, hkv, d = pool_k.shape
    kenc = np.zeros((B, pmax, hkv, d), dtype=np.float64)
    venc = np.zeros((B, pmax, hkv, d), dtype=np.float64)
    for b in range(B):
        for j in range(int(prompt_len[b])):
            page = int(page_table[b, j // page_size])
            kenc[b, j] = pool_k[page, j % page_size]
            venc[b, j] = pool_v[page, j % page_size]
    return kenc, venc


def attn_decode(q, kc, vc, kenc, venc, prompt_len, window):
    """Decoder-mode attention of the canvas over prompt KV and a +-W canvas window.

    24-ai.news, "How does diffusion text generation differ?": decoder mode uses
    bidirectional attention within a sliding window of +-W tokens over the
    canvas.  thakicloud.com, "What is DiffusionGemma": decoder mode reads the
    encoder-mode (causal) KV cache of the prompt.

    Readings: the window is inclusive, |i - j| <= W, clipped at the canvas
    edges, self included; every prompt key is visible to every canvas row; one
    softmax runs jointly over prompt keys and window keys; the score scale is
    1/sqrt(d_head) with no softcap; query head h reads KV head h // (Hq/Hkv).

    q: [B, C, Hq, d]; kc, vc: [B, C, Hkv, d]; kenc, venc: [B, Pmax, Hkv, d];
    prompt_len: [B].  Returns out [B, C, Hq, d] and lse [B, Hq, C] (natural log).
    """
    q = np.asarray(q, dtype=np.float64)
    B, C, hq, d = q.shape
    hkv = kc.shape[2]
    group = hq // hkv
    scale = 1.0 / np.sqrt(d)
    pos = np.arange(C)
    canvas_mask = np.abs(pos[:, None] - pos[None, :]) <= window  # [C, C]
    out = np.zeros((B, C, hq, d), dtype=np.float64)
    lse = np.zeros((B, hq, C), dtype=np.float64)
    for b in range(B):
        P = int(prompt_len[b])
        for h in range(hq):
            g = h // group
            keys = np.concatenate([np.asarray(kenc[b, :P, g], np.float64),
                                   np.asarray(kc[b, :, g], np.float64)], axis=0)
            vals = np.concatenate([np.asarray(venc[b, :P, g], np.float64),
                                   np.asarray(vc[b, :, g], np.float64)], axis=0)
            s = (q[b, :, h] @ keys.T) * scale  # [C, P + C]
            mask = np.concatenate([np.ones((C, P), dtype=bool), canvas_mask], axis=1)
            s = np.where(mask, s, NEG_INF)
            m = s.max(axis=1, keepdims=True)
            ex = np.exp(s - m)
            tot = ex.sum(axis=1, keepdims=True)
            out[b, :, h] = (ex / tot) @ vals
            lse[b, h] = (m + np.log(tot))[:, 0]
    return out, lse


def prefill_attn(q, k, v, prompt_len, rows=None):
    """Encoder-mode attention of each request's prompt over itself, causally.

    thakicloud.com, "What is DiffusionGemma": the one backbone also runs in an
    encoder mode that reads the prompt causally and keeps its KV cache for the
    decoder mode.  24-ai.news, "How does diffusion text generation differ?":
    the encoder mode is causal.

    Readings: row i of request b sees keys j <= i of the same request (self
    included); scale 1/sqrt(d_head), no softcap; query head h reads KV head
    h // (Hq/Hkv); rows at or past prompt_len[b] are not computed (left zero,
    lse 0).  ``rows`` (optional) limits the work to those row indices.

    q: [B, P, Hq, d]; k, v: [B, P, Hkv, d]; prompt_len: [B].
    Returns out [B, P, Hq, d] and lse [B, Hq, P] (natural log).
    """
    q = np.asarray(q, dtype=np.float64)
    B, P, hq, d = q.shape
    hkv = k.shape[2]
    group = hq // hkv
    scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, P, hq, d), dtype=np.float64)
    lse = np.zeros((B, hq, P), dtype=np.float64)
    for b in range(B):
        n = int(min(max(int(prompt_len[b]), 0), P))
        idx = np.arange(n) if rows is None else np.array([r for r in rows if r < n], np.int64)
        if idx.size == 0:
            continue
        last = int(idx.max()) + 1
        for h in range(hq):
            g = h // group
            keys = np.asarray(k[b, :last, g], np.float64)
            vals = np.asarray(v[b, :last, g], np.float64)
            s = (q[b, idx, h] @ keys.T) * scale                 # [rows, last]
            s = np.where(np.arange(last)[None, :] <= idx[:, None], s, NEG_INF)
            m = s.max(axis=1, keepdims=True)
            ex = np.exp(s - m)
            tot = ex.sum(axis=1, keepdims=True)
            out[b, idx, h] = (ex / tot) @ vals
            lse[b, h, idx] = (m + np.log(tot))[:, 0]
    return out, lse


def attn_mixed(mode, rows_len, q, kc, vc, kenc, venc, prompt_len, window):
    """Encoder- and decoder-mode requests of one batch, each by its own definition.

    24-ai.news, "DiffusionGemma integrated into vLLM" ("Integration into the vLLM
    infrastructure"): causal attention switched per sequence lets encoder-mode
    and decoder-mode requests share a batch.

    Request b with mode[b] = 0 is ``attn_decode`` of its first rows_len[b] rows
    (the canvas) over its prompt KV; mode[b] = 1 is ``prefill_attn`` of its first
    rows_len[b] rows.  Rows past rows_len[b] are left zero (lse 0).
    q: [B, C, Hq, d]; kc, vc: [B, C, Hkv, d]; kenc, venc: [B, Pmax, Hkv, d].
    """
    B, C, hq, d = q.shape
    out = np.zeros((B, C, hq, d), dtype=np.float64)
    lse = np.zeros((B, hq, C), dtype=np.float64)
    for b in range(B):
        n = int(min(max(int(rows_len[b]), 0), C))
        if n == 0:
            continue
        if int(mode[b]):
            o, l = prefill_attn(q[b:b + 1, :n], kc[b:b + 1, :n], vc[b:b + 1, :n], [n])
        else:
            o, l = attn_decode(q[b:b + 1, :n], kc[b:b + 1, :n], vc[b:b + 1, :n],
                               kenc[b:b + 1], venc[b:b + 1], prompt_len[b:b + 1], window)
        out[b, :n] = o[0]
        lse[b, :, :n] = l[0]
    return out, lse


def paged_write(k, v, prompt_len, page_table, page_size, n_pages):
    """The page pools an encoder prefill leaves behind: row i of request b goes to
    pool[page_table[b, i // page_size], i % page_size] for i < prompt_len[b]
    (the inverse of ``paged_to_contiguous``).  Untouched pool rows stay zero.

    k, v: [B, P, Hkv, d].  Returns pool_k, pool_v [n_pages, page_size, Hkv, d].
    """
    B, P, hkv, d = k.shape
    pool_k = np.zeros((n_pages, page_size, hkv, d), dtype=np.float64)
    pool_v = np.zeros_like(pool_k)
    for b in range(B):
        for i in range(int(min(max(int(prompt_len[b]), 0), P))):
            pg = int(page_table[b, i // page_size])
            pool_k[pg, i % page_size] = k[b, i]
            pool_v[pg, i % page_size] = v[b, i]
    return pool_k, pool_v


# --------------------------------------------------------------------------
# a2: lm-head -> log-softmax -> entropy
# --------------------------------------------------------------------------
def _logits(h, w, inv_t):
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    return (h @ w.T) * np.asarray(inv_t, dtype=np.float64)[:, None]


def lmhead_stats(h, w, inv_t):
    """Per-row log-normaliser, entropy, max logit and argmax of softmax(h W^T / T).

    tau-home.com, "Refusing JSON token generation": the read takes logprobs and
    entropy from one denoise forward.  24-ai.news, "Token commit mechanism":
    each token's confidence comes from this distribution.

    Readings: temperature divides the logits before the softmax (z = h.w / T);
    entropy is in nats, H = lse - sum_v p_v z_v; argmax ties go to the lowest id.

    h: [M, D]; w: [V, D]; inv_t: [M].  Returns (lse, entropy, maxz, argmax).
    """
    z = _logits(h, w, inv_t)
    m = z.max(axis=1)
    ex = np.exp(z - m[:, None])
    tot = ex.sum(axis=1)
    lse = m + np.log(tot)
    p = ex / tot[:, None]
    ent = lse - (p * z).sum(axis=1)
    arg = np.argmax(z, axis=1)  # first occurrence = lowest id on ties
    return lse, ent, m, arg.astype(np.int64)


def label_logits(h, w, inv_t, label_ids, n_labels):
    """Scaled logits of the allowed labels: z[s, k] = (h_s . w[label_{s,k}]) / T_s.

    h: [S, D] rows being read; label_ids: [S, Kmax] (entries past n_labels ignored).
    Returns [S, Kmax] with NaN past n_labels.
    """
    S, kmax = label_ids.shape
    out = np.full((S, kmax), np.nan)
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    for s in range(S):
        n = int(n_labels[s])
        ids = np.asarray(label_ids[s, :n], dtype=np.int64)
        out[s, :n] = (w[ids] @ h[s]) * float(inv_t[s])
    return out


# --------------------------------------------------------------------------
# a0 + a3: noise draws and the slot read
# --------------------------------------------------------------------------
def slot_noise_rows(h, e, slot_row, slot_req, seed, step, n_draws, vocab):
    """Noised hidden rows of every (slot, draw).

    sotaaz.com, "The server accepts at most 26 alternatives per question": the
    answer slot is left as noise and the server re-reads it with fresh noise
    draws.  Reading (no model exists here): draw r of slot s reads the hidden
    row h[slot_row[s]] + E[n], with n the Philox noise token for counter
    (slot_req[s], step, r, s); draw 0 is noised too.  The sum is formed in fp32
    and rounded to bf16, as the GPU's GEMM operand is.

    Returns rows [S * n_draws, D] ordered (slot-major, draw-minor) and tokens
    [S, n_draws].
    """
    S = len(slot_row)
    D = h.shape[1]
    rows = np.zeros((S * n_draws, D), dtype=np.float32)
    toks = np.zeros((S, n_draws), dtype=np.int64)
    for s in range(S):
        t = noise_tokens(seed, int(slot_req[s]), step, n_draws, S, vocab)[:, s]
        toks[s] = t
        for r in range(n_draws):
            acc = np.asarray(h[slot_row[s]], np.float32) + np.asarray(e[t[r]], np.float32)
            rows[s * n_draws + r] = bf16_round(acc)
    return rows, toks


def _entropy(q):
    q = np.asarray(q, dtype=np.float64)
    nz = q > 0
    return float(-(q[nz] * np.log(q[nz])).sum())


def slot_read(z_lab, lse_draw, n_labels, samples, gate):
    """Renormalised label distribution, entropy, gated resample and choice per slot.

    tau-home.com, "Refusing JSON token generation": read the logprobs of the
    slot's allowed label ids and the entropy.  sotaaz.com, "The server accepts
    at most 26 alternatives per question": if the first read's entropy exceeds
    0.1, each stage is read four times and averaged; ``samples: 1`` keeps one
    read.

    Readings: ``samples`` is the total number of reads per stage, read 0 being
    the gate; the gate is strict (H0 > gate) on the renormalised label entropy
    of read 0; the average is the arithmetic mean of the per-read label
    distributions q^(r); the answer is argmax of the average (ties to the
    lowest label index); the reported entropy is that of the average.

    z_lab: [S, R, Kmax] label logits of each draw (NaN past n_labels);
    lse_draw: [S, R] full-vocabulary log-normaliser of each draw row.
    Returns dict with q_avg [S, Kmax], h_slot [S], chosen [S], lp [S, R, Kmax],
    resampled [S] (0/1), n_reads [S], h_draw [S, R].
    """
    S, R, kmax = z_lab.shape
    q_avg = np.zeros((S, kmax))
    h_slot = np.zeros(S)
    chosen = np.zeros(S, dtype=np.int64)
    resampled = np.zeros(S, dtype=np.int64)
    n_reads = np.zeros(S, dtype=np.int64)
    lp = np.full((S, R, kmax), np.nan)
    h_draw = np.zeros((S, R))
    for s in range(S):
        n = int(n_labels[s])
        if n == 0:  # a question whose ask_if did not fire: not read
            chosen[s] = -1
            lp[s] = 0.0
            continue
        qs = []
        for r in range(R):
            z = np.asarray(z_lab[s, r, :n], np.float64)
            lp[s, r, :n] = z - lse_draw[s, r]
            m = z.max()
            ex = np.exp(z - m)
            q = ex / ex.sum()
            qs.append(q)
            h_draw[s, r] = _entropy(q)
        if samples > 1 and h_draw[s, 0] > gate:
            qbar = np.mean(np.stack(qs[:samples]), axis=0)
            resampled[s] = 1
            n_reads[s] = samples
        else:
            qbar = qs[0]
            n_reads[s] = 1
        q_avg[s, :n] = qbar
        chosen[s] = int(np.argmax(qbar))
        h_slot[s] = _entropy(qbar)
    return dict(q_avg=q_avg, h_slot=h_slot, chosen=chosen, lp=lp,
                resampled=resampled, n_reads=n_reads, h_draw=h_draw)


def ask_if_fires(stage1_chosen, ask_if_value):
    """sotaaz.com, "The server accepts at most 26 alternatives per question":
    a question carrying ``ask_if`` is read only when the earlier answer matches."""
    return int(stage1_chosen) == int(ask_if_value)


def ask_if_select(chosen1, cond_slot, cond_value, q_owner, q_label_ids, q_n_labels, S2):
    """Stage-2 slot table from the stage-1 answers (same page and section).

    Question q asks its labels at stage-2 slot q_owner[q] if the stage-1 answer
    of slot cond_slot[q] equals cond_value[q].  Reading: when several fired
    questions own one slot the first (lowest q) is read; a slot with none is not
    asked (n_labels 0).  Returns label_ids2 [S2, 26] (-1 padded), n_labels2 [S2],
    fired [Q].
    """
    Q = len(cond_slot)
    fired = np.array([1 if 0 <= cond_slot[q] < len(chosen1)
                      and ask_if_fires(chosen1[cond_slot[q]], cond_value[q]) else 0
                      for q in range(Q)], dtype=np.int64)
    label_ids2 = np.full((S2, 26), -1, dtype=np.int64)
    n_labels2 = np.zeros(S2, dtype=np.int64)
    for j in range(S2):
        for q in range(Q):
            if q_owner[q] == j and fired[q]:
                n = int(q_n_labels[q])
                n_labels2[j] = n
                label_ids2[j, :n] = q_label_ids[q, :n]
                break
    return label_ids2, n_labels2, fired


# --------------------------------------------------------------------------
# a4: entropy-ordered commit
# --------------------------------------------------------------------------
def commit(entropy, argmax, cand, gamma):
    """Accept the most confident open positions until cumulative entropy passes gamma.

    24-ai.news, "Token commit mechanism": each step computes every token's
    confidence and accepts tokens from the most confident down until the
    cumulative entropy exceeds a preset threshold.

    Readings: confidence is low entropy, so candidates are ordered by entropy
    ascending with ties to the lower position; the first candidate is always
    accepted (the loop must progress) and the k-th is accepted while the sum of
    the first k entropies stays <= gamma (inclusive); the committed token is
    the row's greedy argmax.

    entropy, argmax, cand: [B, C]; gamma: [B].  Returns commit (0/1) [B, C],
    tokens [B, C] (argmax where committed, -1 elsewhere), n_commit [B].
    """
    entropy = np.asarray(entropy, dtype=np.float64)
    B, C = entropy.shape
    out = np.zeros((B, C), dtype=np.int64)
    toks = np.full((B, C), -1, dtype=np.int64)
    n = np.zeros(B, dtype=np.int64)
    for b in range(B):
        idx = [i for i in range(C) if cand[b, i]]
        idx.sort(key=lambda i: (entropy[b, i], i))
        total = 0.0
        for k, i in enumerate(idx):
            total += entropy[b, i]
            if k > 0 and total > gamma[b]:
                break
            out[b, i] = 1
            toks[b, i] = int(argmax[b, i])
            n[b] += 1
    return out, toks, n


# --------------------------------------------------------------------------
# a5: self-conditioning expected embedding
# --------------------------------------------------------------------------
def selfcond_embed(h, w, e, inv_t):
    """Probability-weighted embedding average e_i = sum_v softmax(z_i)_v E[v].

    24-ai.news, "Token commit mechanism": between steps the previous step's
    full softmax is turned into a probability-weighted average of embeddings
    and fed back as an extra input.  Same temperature reading as lmhead_stats.
    """
    z = _logits(h, w, inv_t)
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    p /= p.sum(axis=1, keepdims=True)
    return p @ np.asarray(e, dtype=np.float64)


# --------------------------------------------------------------------------
# a6: the multi-step loop
# --------------------------------------------------------------------------
def canvas_update(h0, e_sc, emb, tokens, committed):
    """Next-step hidden rows: h0 + e for open rows, h0 + E[token] for committed rows.

    24-ai.news, "Token commit mechanism" says the expected embedding is fed as
    an extra input; the plainest additive reading is used.  The fp32 sum is
    rounded to bf16 because it is the next lm-head GEMM's operand.
    h0, e_sc: [M, D]; tokens: [M] (ignored where not committed); committed: [M].
    """
    h0 = np.asarray(h0, dtype=np.float32)
    add = np.asarray(e_sc, dtype=np.float32).copy()
    for i in np.nonzero(np.asarray(committed))[0]:
        add[i] = np.asarray(emb[int(tokens[i])], dtype=np.float32)
    return bf16_round(h0 + add)


def denoise_loop(h0, w, e, inv_t, cand0, gamma, n_steps):
    """Run the lm-head -> commit -> self-conditioning loop for one request.

    24-ai.news, "How does diffusion text generation differ?" and "Token commit
    mechanism": the canvas is refined over several steps; committed tokens are
    fixed and leave the candidate set; self-conditioning feeds the next step.
    Returns the per-step records (entropy, argmax, commit, tokens, e) and the
    final committed mask and tokens.
    """
    C = h0.shape[0]
    cand = np.asarray(cand0, dtype=bool).copy()
    committed = np.zeros(C, dtype=bool)
    tokens = np.full(C, -1, dtype=np.int64)
    h = np.asarray(h0, dtype=np.float32)
    steps = []
    for _ in range(n_steps):
        lse, ent, maxz, arg = lmhead_stats(h, w, inv_t)
        cm, tk, n = commit(ent[None], arg[None], cand[None], np.array([gamma]))
        new = cm[0].astype(bool)
        tokens[new] = tk[0][new]
        committed |= new
        cand &= ~new
        e_sc = selfcond_embed(h, w, e, inv_t)
        steps.append(dict(lse=lse, entropy=ent, maxz=maxz, argmax=arg,
                          commit=cm[0], tokens=tk[0], n_commit=int(n[0]), e=e_sc))
        h = canvas_update(h0, e_sc, e, tokens, committed)
    return steps, committed, tokens
