"""Margin enforcement for parity inputs (uses the oracle; test infrastructure).

Decisions (chosen label, resample gate, commit set, committed argmax) are
compared bit-exact, so the inputs are re-drawn until every decision is at
least a margin away from its threshold in the oracle's float64 arithmetic:
  |H0 - gate| > 4e-3 nats, top-2 gap of the averaged label distribution
  > 1e-4, entropy gaps around the commit cut > 4e-3 and |S_k - gamma| > 4e-3 k,
  full-vocabulary top-2 logit gap > 1e-3 on committed rows.
"""
import numpy as np

import oracle
from structured_slot_reads_gb300 import inputs

GATE_MARGIN = 4e-3
CHOICE_MARGIN = 1e-4
COMMIT_MARGIN = 4e-3
ARGMAX_MARGIN = 1e-3


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
                     samples, gate, lse_rows=None):
    rows, toks = oracle.slot_noise_rows(h, e, slot_row, slot_req, seed, step, samples, w.shape[0])
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


def slot_margins_ok(res, n_labels, gate):
    for s in range(len(n_labels)):
        if abs(res["h_draw"][s, 0] - gate) <= GATE_MARGIN:
            return False
        q = np.sort(res["q_avg"][s, : n_labels[s]])
        if len(q) > 1 and q[-1] - q[-2] <= CHOICE_MARGIN:
            return False
    return True


def prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, step,
                        samples, gate, modes, max_attempts=30):
    """Plant each slot's mode, re-drawing its hidden row until the margins hold."""
    h = h.copy()
    for attempt in range(max_attempts):
        for s, r in enumerate(slot_row):
            if modes[s] is not None:
                h[r] = plant(h[r], w, inv_t[r], label_ids[s], modes[s])
        res = slot_read_oracle(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed,
                               step, samples, gate)
        if slot_margins_ok(res, n_labels, gate):
            return h, res
        h = inputs.redraw_rows(h, slot_row, seed, attempt + 1)
    raise RuntimeError("could not meet slot margins")


def commit_margins_ok(ent, cand, gamma, z=None, arg_rows=None):
    """Commit cut and (optionally) argmax margins for one request."""
    idx = [i for i in range(len(ent)) if cand[i]]
    idx.sort(key=lambda i: (ent[i], i))
    if not idx:
        return True
    e = np.array([ent[i] for i in idx])
    if len(e) > 1 and np.min(np.diff(e)) <= COMMIT_MARGIN:
        # only the gaps near the cut matter; check them all for simplicity on small canvases
        cs = np.cumsum(e)
        k = int(np.searchsorted(cs, gamma, side="right"))
        lo, hi = max(0, k - 2), min(len(e) - 1, k + 2)
        if np.any(np.diff(e[lo:hi + 1]) <= COMMIT_MARGIN):
            return False
    cs = np.cumsum(e)
    ks = np.arange(1, len(e) + 1)
    if np.any(np.abs(cs - gamma) <= COMMIT_MARGIN * ks):
        return False
    return True
