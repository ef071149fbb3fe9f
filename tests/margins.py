"""Margin enforcement for parity inputs (uses the oracle; test infrastructure).

Decisions (chosen label, resample gate, commit set, committed argmax) are
compared bit-exact, so the inputs are re-drawn until every decision is at
least a margin away from its threshold in the oracle's float64 arithmetic:
  |H0 - gate| > 4e-3 nats;
  log-ratio of the top two probabilities of the averaged label distribution
    > 1e-3: for one read ln(q1/q2) is the top-2 label-logit gap itself, and an
    average of reads has relative errors no larger than its reads' logit
    errors, so the same bound holds for it;
  the commit set: the entropy gap between the last accepted and the first
    refused candidate > 4e-3, and the prefix sums on either side of the cut
    at least 4e-3 k from gamma (no other order or sum can change the set);
  full-vocabulary top-2 logit gap > 1e-3 on committed rows.
The fp32 error these guard against is about 1e-4 (a 2816-long bf16 dot
product accumulated in fp32).
"""
import numpy as np

import oracle
from structured_slot_reads_gb300 import inputs

GATE_MARGIN = 4e-3
CHOICE_MARGIN = 1e-3
COMMIT_MARGIN = 4e-3
ARGMAX_MARGIN = 1e-3


def _top2_gap(z):
    part = np.partition(z, -2, axis=1)
    return part[:, -1] - part[:, -2]


def plant(h_row, w, inv_t_row, label_ids, mode):
    """Make a slot row's first read high-entropy ('high') or dominated by label 0 ('low')."""
    x = np.asarray(h_row, np.float64)
    if mode == "high":
        x = x / 4.0
    elif mode == "low":
        wl = np.asarray(w[label_ids[0]], np.float64)
        x = x + (12.0 / float(inv_t_row)) * wl / np.dot(wl, wl)
    return inputs.to_bf16(x.astype(np.float32))


def slot_read_oracle(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, step,
                     samples, gate, lse_rows=None, sel=None):
    """The oracle's read of a slot table.  ``sel`` (optional) reads only those slots
    of the table, each with its noise draws of the whole table (the Philox counter
    holds the slot's index in the table), so large tables can be sampled."""
    rows, toks = oracle.slot_noise_rows(h, e, slot_row, slot_req, seed, step, samples, w.shape[0])
    if sel is not None:
        sel = np.asarray(sel, dtype=np.int64)
        rows = rows[(sel[:, None] * samples + np.arange(samples)[None, :]).reshape(-1)]
        toks = toks[sel]
        slot_row, label_ids, n_labels = slot_row[sel], label_ids[sel], n_labels[sel]
    inv_rows = np.repeat(inv_t[slot_row], samples)
    if lse_rows is None:
        lse_rows, _, _, _ = oracle.lmhead_stats(rows, w, inv_rows)
    S = len(slot_row)
    zl = oracle.label_logits(rows, w, inv_rows, np.repeat(label_ids, samples, axis=0),
                             np.repeat(n_labels, samples))
    z = zl.reshape(S, samples, -1)
    out = oracle.slot_read(z, lse_rows.reshape(S, samples), n_labels, samples, gate)
    out["tokens"] = toks
    out["rows"] = rows
    return out


def slot_ok(res, n_labels, s, gate):
    """Slot s's gate and choice are a margin away from changing (a slot that was
    not asked, with no labels, has no decision)."""
    n = int(n_labels[s])
    if n == 0:
        return True
    if abs(res["h_draw"][s, 0] - gate) <= GATE_MARGIN:
        return False
    q = np.sort(res["q_avg"][s, :n])
    return n == 1 or (q[-2] <= 0 and q[-1] > 0) or np.log(q[-1] / q[-2]) > CHOICE_MARGIN


def slot_margins_ok(res, n_labels, gate):
    return all(slot_ok(res, n_labels, s, gate) for s in range(len(n_labels)))


def prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, step,
                        samples, gate, modes, max_attempts=30, sel=None):
    """Plant each slot's mode, re-drawing its hidden row until the margins hold.
    With ``sel`` only those slots of the table are planted, read and re-drawn
    (``modes`` then has one entry per selected slot)."""
    h = h.copy()
    idx = np.arange(len(slot_row)) if sel is None else np.asarray(sel, dtype=np.int64)
    for attempt in range(max_attempts):
        for j, s in enumerate(idx):
            r = slot_row[s]
            if modes[j] is not None:
                h[r] = plant(h[r], w, inv_t[r], label_ids[s], modes[j])
        res = slot_read_oracle(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed,
                               step, samples, gate, sel=sel)
        if slot_margins_ok(res, n_labels[idx], gate):
            return h, res
        h = inputs.redraw_rows(h, slot_row[idx], seed, attempt + 1)
    raise RuntimeError("could not meet slot margins")


def commit_margins_ok(ent, cand, gamma, z=None, arg_rows=None):
    """The commit set of one request is a margin away from changing.

    Candidates sorted by (entropy, position); the first is always accepted and
    the k-th while S_k <= gamma, so n = max(1, #{k : S_k <= gamma}) are taken.
    The set changes only if the last accepted and the first refused candidate
    swap places, or if S_n (n >= 2) rises above gamma, or S_{n+1} falls below it.
    """
    idx = [i for i in range(len(ent)) if cand[i]]
    idx.sort(key=lambda i: (ent[i], i))
    if not idx:
        return True
    e = np.array([ent[i] for i in idx], dtype=np.float64)
    cs = np.cumsum(e)
    n = max(1, int(np.searchsorted(cs, gamma, side="right")))
    if n >= 2 and gamma - cs[n - 1] <= COMMIT_MARGIN * n:
        return False
    if n < len(e):
        if e[n] - e[n - 1] <= COMMIT_MARGIN:
            return False
        if cs[n] - gamma <= COMMIT_MARGIN * (n + 1):
            return False
    return True


def two_stage_oracle(h, w, e, inv_t, slots1, questions, slots2, seed, samples, gate):
    """Oracle of a two-stage read: stage 1 at step 0, the ask_if table from its
    choices, stage 2 (its asked slots) at step 1.

    slots1 = (rows, reqs, label_ids, n_labels); questions = (cond_slot,
    cond_value, owner, label_ids, n_labels); slots2 = (rows, reqs).
    Returns (stage-1 result, (label_ids2, n_labels2, fired), stage-2 result).
    """
    rows1, req1, lab1, n1 = slots1
    st1 = slot_read_oracle(h, w, e, inv_t, rows1, req1, lab1, n1, seed, 0, samples, gate)
    cs, cv, own, qlab, qn = questions
    rows2, req2 = slots2
    lab2, n2, fired = oracle.ask_if_select(st1["chosen"], cs, cv, own, qlab, qn, len(rows2))
    st2 = slot_read_oracle(h, w, e, inv_t, rows2, req2, lab2, n2, seed, 1, samples, gate)
    return st1, (lab2, n2, fired), st2


def prepare_two_stage_inputs(h, w, e, inv_t, slots1, questions, slots2, seed, samples, gate,
                             max_attempts=30):
    """Re-draw the hidden rows of the slots whose decision (stage 1, or the stage-2
    slot a request asks) is too close to its threshold, until every decision of
    both stages has its margin.  Returns (h, oracle result as two_stage_oracle)."""
    h = h.copy()
    rows1, rows2 = slots1[0], slots2[0]
    for attempt in range(max_attempts):
        st1, t2, st2 = two_stage_oracle(h, w, e, inv_t, slots1, questions, slots2, seed, samples,
                                        gate)
        bad = [int(rows1[s]) for s in range(len(rows1)) if not slot_ok(st1, slots1[3], s, gate)]
        bad += [int(rows2[j]) for j in range(len(rows2)) if not slot_ok(st2, t2[1], j, gate)]
        if not bad:
            return h, (st1, t2, st2)
        h = inputs.redraw_rows(h, sorted(set(bad)), seed, attempt + 1)
    raise RuntimeError("could not meet two-stage slot margins")


def prepare_loop_inputs(shape, n_steps, seed=0, max_attempts=60):
    """Inputs of an n-step loop whose every decision has its margin in the oracle's
    float64 arithmetic: each step's commit set, the argmax of every row it commits,
    and each step's slot reads (read from that step's canvas input).  Re-draws the
    hidden rows until all hold.  Returns (x, oracle steps, per-step slot reads)."""
    x = inputs.step_inputs(shape, seed)
    w64 = x["w"].astype(np.float64)
    for attempt in range(max_attempts):
        steps, _, _ = oracle.denoise_loop(x["h"], w64, x["e"], x["inv_t"],
                                          x["cand"][0].astype(bool), shape.gamma, n_steps)
        ok = True
        cand = x["cand"][0].astype(bool).copy()
        committed = np.zeros(shape.C, dtype=bool)
        tokens = np.full(shape.C, -1, dtype=np.int64)
        h = x["h"]
        reads = []
        for t, st in enumerate(steps):
            ok &= commit_margins_ok(st["entropy"], cand, shape.gamma)
            new = st["commit"].astype(bool)
            if new.any():
                z = (h[new].astype(np.float64) @ w64.T) * x["inv_t"][new][:, None]
                ok &= bool(np.all(_top2_gap(z) > ARGMAX_MARGIN))
            if len(shape.slots):
                rd = slot_read_oracle(h, w64, x["e"], x["inv_t"], x["slot_row"],
                                      x["slot_req"], x["label_ids"], x["n_labels"], 0, t,
                                      shape.R, shape.gate)
                ok &= slot_margins_ok(rd, x["n_labels"], shape.gate)
                reads.append(rd)
            if not ok:
                break
            cand &= ~new
            committed |= new
            tokens[new] = st["tokens"][new]
            h = oracle.canvas_update(x["h"], st["e"], x["e"], tokens, committed)
        if ok:
            return x, steps, reads
        x["h"] = inputs.hidden(shape.B * shape.C, shape.D, seed, attempt + 1)
    raise RuntimeError("margins not met")
