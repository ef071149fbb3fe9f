"""Batched two-stage structured reads over a paged prompt KV cache, through libdg.

sotaaz.com, "The server accepts at most 26 alternatives per question": 77
intents do not fit one question (A-Z), so a 9-way group question is read
first and the chosen group's item question (carrying ``ask_if``) second; each
stage re-reads a slot four times when its first read's entropy exceeds 0.1.
One ``TwoStageRead.run`` is, for every request of the batch:

  dg_attn_decode      decoder attention of the canvas over its paged prompt KV
  dg_slot_noise       noised draw rows of stage 1 (group slot + 0-3 other
                      slots) and of stage 2 (the item slot), each stage with
                      its own step index in the Philox counter
  dg_lmhead_logsoftmax_entropy
                      one W pass over the draw rows of both stages: their
                      full-vocabulary lse does not depend on which labels a
                      slot is read with, so stage 2 needs no pass of its own
  dg_slot_finish      stage 1: label logits, renormalise, gate, average
  dg_ask_if_select    stage-2 slot table from the stage-1 answers (on device)
  dg_slot_finish      stage 2, with the labels of the question that fired

This is dg_slot_read for each stage (noise, one W pass, finish) with the two
W passes made one.

Torch allocates every buffer; the library only enqueues work.
"""
import numpy as np
import torch

from . import dg, inputs
from .step import as_stream


def _dev(a, dtype, device):
    return torch.as_tensor(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def _pad26(lab):
    """A label list as one row of a 26-wide table (-1 padded).  A longer list keeps
    only its first 26 ids here; its count still says how many it had, so the slot
    table check refuses it."""
    pad = np.full(dg.MAX_LABELS, -1, np.int32)
    k = min(len(lab), dg.MAX_LABELS)
    pad[:k] = np.asarray(lab)[:k]
    return pad


def slot_outputs(S, R, dev, L=dg.MAX_LABELS):
    """Device buffers of one slot read over S slots with R reads each (label stride L)."""
    f32, i32, u8 = torch.float32, torch.int32, torch.uint8
    return dict(q_avg=torch.empty((S, L), dtype=f32, device=dev),
                h_slot=torch.empty(S, dtype=f32, device=dev),
                chosen=torch.empty(S, dtype=i32, device=dev),
                lp=torch.empty((S, R, L), dtype=f32, device=dev),
                resampled=torch.empty(S, dtype=u8, device=dev),
                n_reads=torch.empty(S, dtype=i32, device=dev),
                tokens=torch.empty((S, R), dtype=i32, device=dev))


class TwoStageRead:
    def __init__(self, shape, w, e, tables, prompt_len, device="cuda", seed=0):
        """tables: inputs.two_stage_tables(shape, seed) (one dict per request)."""
        self.shape = shape
        self.dims = dg.dims_of(shape)
        self.dims.P_max = int(max(prompt_len))      # the page table covers the longest prompt
        self.device = device
        self.w, self.e = w, e
        self.seed = seed
        B, C, D = shape.B, shape.C, shape.D
        bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8
        self.M = B * C
        self.h = torch.empty((self.M, D), dtype=bf, device=device)
        self.inv_t = torch.empty(self.M, dtype=f32, device=device)
        self.q = torch.empty((B, C, shape.Hq, shape.d_head), dtype=bf, device=device)
        self.kc = torch.empty((B, C, shape.Hkv, shape.d_head), dtype=bf, device=device)
        self.vc = torch.empty_like(self.kc)
        self.prompt_len = _dev(prompt_len, i32, device)
        ps = shape.page_size
        self.pages_per_req = int(max((int(p) + ps - 1) // ps for p in prompt_len))
        self.attn_out = torch.empty_like(self.q)
        self.attn_lse = torch.empty((B, shape.Hq, C), dtype=f32, device=device)
        # stage 1: group slot then the other slots of every request
        rows, reqs, labs, ns, self.group_slot = [], [], [], [], []
        for b, t in enumerate(tables):
            self.group_slot.append(len(rows))
            for pos, lab in [(t["group_pos"], t["group_labels"])] + list(t["others"]):
                rows.append(b * C + pos)
                reqs.append(b)
                labs.append(_pad26(lab))
                ns.append(len(lab))
        self.S1 = len(rows)
        # the 26-alternative limit and the label checks, before anything reaches the GPU
        dg.validate_slot_table(self.dims, rows, np.stack(labs), ns, self.M, "stage-1 slot table")
        self.slot_row1 = _dev(rows, i32, device)
        self.slot_req1 = _dev(reqs, i32, device)
        self.label_ids1 = _dev(np.stack(labs), i32, device)
        self.n_labels1 = _dev(ns, i32, device)
        self.host_slots1 = (np.array(rows, np.int32), np.stack(labs), np.array(ns, np.int32))
        # stage-2 questions: one per (request, group option), ask_if = that option
        cs, cv, own, qlab, qn = [], [], [], [], []
        for b, t in enumerate(tables):
            for g, items in enumerate(t["item_labels"]):
                cs.append(self.group_slot[b])
                cv.append(g)
                own.append(b)
                qlab.append(_pad26(items))
                qn.append(len(items))
        self.Q = len(cs)
        # every stage-2 question is checked as a slot of its owner's item row
        item_rows = [b * C + tables[b]["item_pos"] for b in own]
        dg.validate_slot_table(self.dims, item_rows, np.stack(qlab), qn, self.M,
                               "stage-2 question table")
        self.cond_slot = _dev(cs, i32, device)
        self.cond_value = _dev(cv, i32, device)
        self.q_owner = _dev(own, i32, device)
        self.q_label_ids = _dev(np.stack(qlab), i32, device)
        self.q_n_labels = _dev(qn, i32, device)
        self.host_questions = (np.array(cs), np.array(cv), np.array(own), np.stack(qlab),
                               np.array(qn))
        self.S2 = B
        self.slot_row2 = _dev([b * C + t["item_pos"] for b, t in enumerate(tables)], i32, device)
        self.slot_req2 = _dev(list(range(B)), i32, device)
        self.label_ids2 = torch.empty((B, dg.MAX_LABELS), dtype=i32, device=device)
        self.n_labels2 = torch.empty(B, dtype=i32, device=device)
        self.fired = torch.empty(self.Q, dtype=u8, device=device)
        R = shape.R
        self.out1 = slot_outputs(self.S1, R, device)
        self.out2 = slot_outputs(self.S2, R, device)
        d = self.dims
        self.ws_attn = torch.empty(max(dg.dg_workspace_bytes(d, dg.DG_WS_ATTN, 0), 256),
                                   dtype=u8, device=device)
        # the draw rows of both stages (stage 1 first) and their statistics
        self.r1 = self.S1 * R
        n = self.r1 + self.S2 * R
        self.draw_rows = torch.empty((n, D), dtype=bf, device=device)
        self.inv_t_draw = torch.empty(n, dtype=f32, device=device)
        self.lse_draw = torch.empty(n, dtype=f32, device=device)
        self.ent_draw = torch.empty(n, dtype=f32, device=device)
        self.maxz_draw = torch.empty(n, dtype=f32, device=device)
        self.arg_draw = torch.empty(n, dtype=i32, device=device)
        self.ws_lm = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, n), dtype=u8,
                                 device=device)

    def set_kv(self, pool_k, pool_v, page_table):
        self.pool_k, self.pool_v = pool_k, pool_v
        self.page_table = page_table
        self.n_pages = pool_k.shape[0]

    def _noise(self, S, slot_row, slot_req, rows, out, step, stream):
        s = self.shape
        dg._check(dg.dg_slot_noise(self.dims, self.h, self.M, self.e, self.inv_t, slot_row,
                                   slot_req, S, s.R, self.seed, step, self.draw_rows[rows],
                                   self.inv_t_draw[rows], out["tokens"], stream), "dg_slot_noise")

    def _finish(self, S, label_ids, n_labels, rows, out, stream):
        s = self.shape
        dg._check(dg.dg_slot_finish(self.dims, self.draw_rows[rows], self.inv_t_draw[rows],
                                    self.lse_draw[rows], self.w, label_ids, n_labels, S, s.R,
                                    s.R, s.gate, out["q_avg"], out["h_slot"], out["chosen"],
                                    out["lp"], out["resampled"], out["n_reads"], stream),
                  "dg_slot_finish")

    def run(self, stream=None):
        """Enqueue attention + both read stages; returns the number of library kernels."""
        dg._check(dg.dg_attn_decode(self.dims, self.q, self.kc, self.vc, self.pool_k,
                                    self.pool_v, self.page_table, self.page_table.shape[1],
                                    self.n_pages, self.shape.page_size, self.prompt_len,
                                    self.attn_out, self.attn_lse, self.ws_attn, stream),
                  "dg_attn_decode")
        st1, st2 = slice(0, self.r1), slice(self.r1, None)
        self._noise(self.S1, self.slot_row1, self.slot_req1, st1, self.out1, 0, stream)
        self._noise(self.S2, self.slot_row2, self.slot_req2, st2, self.out2, 1, stream)
        dg._check(dg.dg_lmhead_logsoftmax_entropy(self.dims, self.draw_rows,
                                                  self.draw_rows.shape[0], self.w,
                                                  self.inv_t_draw, None, None, None, 0,
                                                  self.lse_draw, self.ent_draw, self.maxz_draw,
                                                  self.arg_draw, None, self.ws_lm, stream),
                  "dg_lmhead_logsoftmax_entropy")
        self._finish(self.S1, self.label_ids1, self.n_labels1, st1, self.out1, stream)
        dg._check(dg.dg_ask_if_select(self.out1["chosen"], self.S1, self.cond_slot,
                                      self.cond_value, self.q_owner, self.q_label_ids,
                                      self.q_n_labels, self.Q, self.S2, self.label_ids2,
                                      self.n_labels2, self.fired, stream), "dg_ask_if_select")
        self._finish(self.S2, self.label_ids2, self.n_labels2, st2, self.out2, stream)
        attn_kernels = 1 if dg.dg_workspace_bytes(self.dims, dg.DG_WS_ATTN, 0) <= 256 else 2
        # noise x 2, one W pass (stats + finalize), finish (label logits + epilogue) x 2,
        # ask_if.  The finishes compute their label logits from the noised rows: the
        # stage-2 labels are known only after stage 1 has been read.
        return attn_kernels + 2 + 2 + 4 + 1

    def decisions(self):
        """Slot decisions completed by one run (stage-1 slots + asked stage-2 slots)."""
        return self.S1 + int((self.n_labels2 > 0).sum().item())

    def check(self, stream=None):
        """Raise dg.DgDeviceError if a kernel of the enqueued runs set a status bit
        (synchronises ``stream``)."""
        return dg.check_status(stream, "two-stage read")


class ReadStep:
    """The read-only step of a structured read (no commit, no self-conditioning).

    tau-home.com, "Refusing JSON token generation": the canvas is prefilled,
    the answer slots are left blank and one denoise forward gives the label
    distribution of every slot.  One ``run`` is dg_attn_decode over the
    contiguous prompt KV plus one dg_slot_read over the slot table of every
    request (the same slots in every request).  The two do not feed each
    other: with ``concurrent=True`` (the default) the attention goes first on a
    side stream, planned for an eighth of the SMs (``dims.sm_share``), and the
    slot read's W pass takes the SMs it leaves.

    ``fp4=True`` reads against an NVFP4 checkpoint (tau-home.com, "Running NVFP4
    locally with a Jev-compatible System One endpoint"): W is quantised once
    (dg_quantize_nvfp4_mma) and the slot read is dg_slot_noise, then the
    block-scaled pass over the S*R draw rows (the rows quantised in the call;
    one gathered label row per draw, which writes z - lse), then dg_slot_finish
    on those gathered values with zero row lse, so that it keeps them as the
    draws' label logprobs.  Slots of up to 26 labels.
    """

    def __init__(self, shape, w, e, device="cuda", seed=0, concurrent=True, fp4=False):
        """Slots with more than 26 labels are read with dg_slot_read_wide (one table of
        stride L = the largest label count)."""
        self.shape = shape
        self.dims = dg.dims_of(shape)
        self.device = device
        self.w, self.e = w, e
        self.seed = seed
        B, C, D = shape.B, shape.C, shape.D
        bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8
        self.M = B * C
        self.h = torch.empty((self.M, D), dtype=bf, device=device)
        self.inv_t = torch.empty(self.M, dtype=f32, device=device)
        self.q = torch.empty((B, C, shape.Hq, shape.d_head), dtype=bf, device=device)
        self.kc = torch.empty((B, C, shape.Hkv, shape.d_head), dtype=bf, device=device)
        self.vc = torch.empty_like(self.kc)
        self.kenc = torch.empty((B, shape.P, shape.Hkv, shape.d_head), dtype=bf, device=device)
        self.venc = torch.empty_like(self.kenc)
        self.prompt_len = torch.full((B,), shape.P, dtype=i32, device=device)
        self.attn_out = torch.empty_like(self.q)
        self.attn_lse = torch.empty((B, shape.Hq, C), dtype=f32, device=device)
        self.L = max([dg.MAX_LABELS] + [k for _, k in shape.slots])
        row, req, lab, n = inputs.slot_table(shape, seed, self.L)
        dg.validate_slot_table(self.dims, row, lab, n, self.M)
        self.S = len(row)
        self.slot_row = _dev(row, i32, device)
        self.slot_req = _dev(req, i32, device)
        self.label_ids = _dev(lab, i32, device)
        self.n_labels = _dev(n, i32, device)
        self.out = slot_outputs(self.S, shape.R, device, self.L)
        self.concurrent = concurrent
        n_sm = dg.dg_num_sms()
        self.dims_side = dg.dims_of(shape, sm_share=max(1, n_sm - n_sm * 7 // 8))
        self._side = None
        self.ws_attn = torch.empty(max(dg.dg_workspace_bytes(self.dims, dg.DG_WS_ATTN, 0),
                                       dg.dg_workspace_bytes(self.dims_side, dg.DG_WS_ATTN, 0),
                                       256), dtype=u8, device=device)
        self.ws_read = torch.empty(dg.dg_workspace_bytes(self.dims, dg.DG_WS_SLOT_READ,
                                                         self.S * shape.R), dtype=u8,
                                   device=device)
        self.fp4 = fp4
        if fp4:
            nd = self.S * shape.R
            if self.L != dg.MAX_LABELS:
                raise ValueError("the NVFP4 read takes slots of at most 26 labels")
            V = shape.V
            self.codes = torch.empty((dg.dg_nvfp4_mma_codes_bytes(V, D),), dtype=u8,
                                     device=device)
            self.sf = torch.empty(((V + 127) // 128, D // 64, 512), dtype=u8, device=device)
            self.g = torch.empty(1, dtype=f32, device=device)
            dg._check(dg.dg_quantize_nvfp4_mma(w, V, D, self.codes, self.sf, self.g),
                      "dg_quantize_nvfp4_mma")
            self.rows_draw = torch.empty((nd, D), dtype=bf, device=device)
            self.inv_t_draw = torch.empty(nd, dtype=f32, device=device)
            self.draw_row = torch.arange(nd, dtype=i32, device=device)
            self.draw_labels = self.label_ids.repeat_interleave(shape.R, dim=0).contiguous()
            self.draw_n = self.n_labels.repeat_interleave(shape.R).contiguous()
            self.lse_draw = torch.empty(nd, dtype=f32, device=device)
            self.zero_lse = torch.zeros(nd, dtype=f32, device=device)
            self.lm = [torch.empty(nd, dtype=f32, device=device) for _ in range(2)]
            self.lm_arg = torch.empty(nd, dtype=i32, device=device)
            self.ws_lm = torch.empty(dg.dg_workspace_bytes(self.dims, dg.DG_WS_LMHEAD_NVFP4_MMA,
                                                           nd), dtype=u8, device=device)

    def run(self, step_idx=0, stream=None):
        """Enqueue attention + the slot read; returns the number of library kernels."""
        s, d, o = self.shape, self.dims, self.out
        main = as_stream(stream)
        attn_stream, attn_dims = main, d
        if self.concurrent:
            if self._side is None:
                self._side = torch.cuda.Stream(device=self.h.device)
            attn_stream, attn_dims = self._side, self.dims_side
            attn_stream.wait_stream(main)
        dg._check(dg.dg_attn_decode(attn_dims, self.q, self.kc, self.vc, self.kenc, self.venc,
                                    None, 0, 0, 0, self.prompt_len, self.attn_out,
                                    self.attn_lse, self.ws_attn, attn_stream), "dg_attn_decode")
        stream = main
        if self.fp4:
            nd = self.S * s.R
            dg._check(dg.dg_slot_noise(d, self.h, self.M, self.e, self.inv_t, self.slot_row,
                                       self.slot_req, self.S, s.R, self.seed, step_idx,
                                       self.rows_draw, self.inv_t_draw, o["tokens"], stream),
                      "dg_slot_noise")
            dg._check(dg.dg_lmhead_logsoftmax_entropy_nvfp4_mma(
                d, self.rows_draw, nd, self.codes, self.sf, self.g, self.inv_t_draw,
                self.draw_row, self.draw_labels, self.draw_n, nd, self.lse_draw, self.lm[0],
                self.lm[1], self.lm_arg, o["lp"], self.ws_lm, stream),
                "dg_lmhead_logsoftmax_entropy_nvfp4_mma")
            dg._check(dg.dg_slot_finish(d, None, None, self.zero_lse, None, self.label_ids,
                                        self.n_labels, self.S, s.R, s.R, s.gate, o["q_avg"],
                                        o["h_slot"], o["chosen"], o["lp"], o["resampled"],
                                        o["n_reads"], stream), "dg_slot_finish")
        elif self.L == dg.MAX_LABELS:
            dg._check(dg.dg_slot_read(d, self.h, self.M, self.w, self.e, self.inv_t,
                                      self.slot_row, self.slot_req, self.label_ids,
                                      self.n_labels, self.S, self.seed, step_idx, s.R, s.gate,
                                      o["q_avg"], o["h_slot"], o["chosen"], o["lp"],
                                      o["resampled"], o["n_reads"], o["tokens"], self.ws_read,
                                      stream), "dg_slot_read")
        else:
            dg._check(dg.dg_slot_read_wide(d, self.h, self.M, self.w, self.e, self.inv_t,
                                           self.slot_row, self.slot_req, self.label_ids,
                                           self.n_labels, self.S, self.L, self.seed, step_idx,
                                           s.R, s.gate, o["q_avg"], o["h_slot"], o["chosen"],
                                           o["lp"], o["resampled"], o["n_reads"], o["tokens"],
                                           self.ws_read, stream), "dg_slot_read_wide")
        if self.concurrent:
            main.wait_stream(attn_stream)
        attn_kernels = 1 if dg.dg_workspace_bytes(attn_dims, dg.DG_WS_ATTN, 0) <= 256 else 2
        if self.fp4:
            # noise; row quantisation (one kernel up to 16 rows, else three), gather
            # table, W pass, finalize; slot epilogue
            return attn_kernels + (6 if self.S * s.R <= 16 else 8)
        # noise, the W pass (gathering the label logits) + finalize, slot epilogue
        return attn_kernels + 4

    def check(self, stream=None):
        """Raise dg.DgDeviceError if a kernel of the enqueued reads set a status bit
        (synchronises ``stream``)."""
        return dg.check_status(stream, "read step")


class Prefill:
    """Encoder-mode prefill of a batch of prompts: causal attention of every prompt over
    itself, its K/V written into a shared page pool (dg_prefill_attn), the layout the
    decoder-mode read takes."""

    def __init__(self, B, P, Hq, Hkv, d_head, page_size=16, device="cuda", seed=0):
        bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8
        self.B, self.P, self.Hq, self.Hkv, self.d = B, P, Hq, Hkv, d_head
        self.dims = dg.make_dims(B=B, P_max=P, Hq=Hq, Hkv=Hkv, d_head=d_head)
        self.q = torch.empty((B, P, Hq, d_head), dtype=bf, device=device)
        self.k = torch.empty((B, P, Hkv, d_head), dtype=bf, device=device)
        self.v = torch.empty_like(self.k)
        self.prompt_len = torch.full((B,), P, dtype=i32, device=device)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((B, Hq, P), dtype=f32, device=device)
        self.page_size = page_size
        table, self.n_pages = inputs.page_table([P] * B, page_size, seed)
        self.page_table = _dev(table, i32, device)
        self.pool_k = torch.empty((self.n_pages, page_size, Hkv, d_head), dtype=bf, device=device)
        self.pool_v = torch.empty_like(self.pool_k)
        self.ws = torch.empty(max(dg.dg_workspace_bytes(self.dims, dg.DG_WS_PREFILL, 0), 256),
                              dtype=u8, device=device)

    def run(self, step_idx=0, stream=None):
        """Enqueue the prefill; returns the number of library kernels."""
        dg._check(dg.dg_prefill_attn(self.dims, self.q, self.k, self.v, self.prompt_len, self.out,
                                     self.lse, self.page_table, self.page_table.shape[1],
                                     self.n_pages, self.page_size, self.pool_k, self.pool_v,
                                     self.ws, stream), "dg_prefill_attn")
        splits = 1 if dg.dg_workspace_bytes(self.dims, dg.DG_WS_PREFILL, 0) <= 256 else 2
        return splits + 1


class LmHead:
    """One lm-head statistics pass over M rows (lse, entropy, max logit, argmax), on bf16
    operands (dg_lmhead_logsoftmax_entropy), on e4m3 operands with per-row scales
    (dg_quantize_rows_e4m3 of the rows, then dg_lmhead_logsoftmax_entropy_fp8), or on
    bf16 rows against NVFP4 weights (dg_lmhead_logsoftmax_entropy_nvfp4), or with rows
    and weights both NVFP4 on the block-scaled kind (fp4_mma: at most 16 rows,
    dg_lmhead_logsoftmax_entropy_nvfp4_mma); W is quantised once, when the object is
    made."""

    def __init__(self, shape, w, M, fp8=False, device="cuda", fp4=False, fp4_mma=False):
        f32, i32, u8 = torch.float32, torch.int32, torch.uint8
        self.shape, self.M, self.fp8, self.fp4, self.fp4_mma = shape, M, fp8, fp4, fp4_mma
        self.dims = dg.make_dims(d_model=shape.D, V=shape.V)
        self.h = torch.empty((M, shape.D), dtype=torch.bfloat16, device=device)
        self.inv_t = torch.empty(M, dtype=f32, device=device)
        self.lse, self.ent, self.maxz = (torch.empty(M, dtype=f32, device=device)
                                         for _ in range(3))
        self.argmax = torch.empty(M, dtype=i32, device=device)
        kind = dg.DG_WS_LMHEAD_NVFP4_MMA if fp4_mma else dg.DG_WS_LMHEAD
        self.ws = torch.empty(dg.dg_workspace_bytes(self.dims, kind, M), dtype=u8, device=device)
        self.w = w
        if fp4_mma:
            D, V = shape.D, shape.V
            self.codes = torch.empty((dg.dg_nvfp4_mma_codes_bytes(V, D),), dtype=u8,
                                     device=device)
            self.sf = torch.empty(((V + 127) // 128, D // 64, 512), dtype=u8, device=device)
            self.g = torch.empty(1, dtype=f32, device=device)
            dg._check(dg.dg_quantize_nvfp4_mma(w, V, D, self.codes, self.sf, self.g),
                      "dg_quantize_nvfp4_mma")
        if fp4:
            D, V = shape.D, shape.V
            self.codes = torch.empty((D // 64, V, 32), dtype=u8, device=device)
            self.scales = torch.empty((D // 64, V, 4), dtype=u8, device=device)
            self.g = torch.empty(1, dtype=f32, device=device)
            dg._check(dg.dg_quantize_nvfp4(w, V, D, self.codes, self.scales, self.g),
                      "dg_quantize_nvfp4")
        if fp8:
            self.w8 = torch.empty((shape.V, shape.D), dtype=u8, device=device)
            self.w_scale = torch.empty(shape.V, dtype=f32, device=device)
            dg._check(dg.dg_quantize_rows_e4m3(w, shape.V, shape.D, self.w8, self.w_scale),
                      "dg_quantize_rows_e4m3")
            self.h8 = torch.empty((M, shape.D), dtype=u8, device=device)
            self.h_scale = torch.empty(M, dtype=f32, device=device)

    def run(self, step_idx=0, stream=None):
        """Enqueue one pass; returns the number of library kernels."""
        d = self.dims
        if self.fp4_mma:
            dg._check(dg.dg_lmhead_logsoftmax_entropy_nvfp4_mma(d, self.h, self.M, self.codes,
                                                                self.sf, self.g, self.inv_t,
                                                                None, None, None, 0, self.lse,
                                                                self.ent, self.maxz,
                                                                self.argmax, None, self.ws,
                                                                stream),
                      "dg_lmhead_logsoftmax_entropy_nvfp4_mma")
            # the rows' quantisation (one kernel up to 16 rows, else amax, quantise
            # and scale), the pass, the finalize
            return (1 if self.M <= 16 else 3) + 2
        if self.fp4:
            dg._check(dg.dg_lmhead_logsoftmax_entropy_nvfp4(d, self.h, self.M, self.codes,
                                                            self.scales, self.g, self.inv_t,
                                                            None, None, None, 0, self.lse,
                                                            self.ent, self.maxz, self.argmax,
                                                            None, self.ws, stream),
                      "dg_lmhead_logsoftmax_entropy_nvfp4")
            return 2
        if not self.fp8:
            dg._check(dg.dg_lmhead_logsoftmax_entropy(d, self.h, self.M, self.w, self.inv_t,
                                                      None, None, None, 0, self.lse, self.ent,
                                                      self.maxz, self.argmax, None, self.ws,
                                                      stream),
                      "dg_lmhead_logsoftmax_entropy")
            return 2
        dg._check(dg.dg_quantize_rows_e4m3(self.h, self.M, self.shape.D, self.h8, self.h_scale,
                                           stream), "dg_quantize_rows_e4m3")
        dg._check(dg.dg_lmhead_logsoftmax_entropy_fp8(d, self.h8, self.h_scale, self.M, self.w8,
                                                      self.w_scale, self.inv_t, None, None, None,
                                                      0, self.lse, self.ent, self.maxz,
                                                      self.argmax, None, self.ws, stream),
                  "dg_lmhead_logsoftmax_entropy_fp8")
        return 3


class Heads:
    """The fused pass of a step alone (statistics of M canvas rows, the normalisers
    of n_draw draw rows, the bf16 self-conditioning probabilities) on bf16
    operands (dg_denoise_heads, W streamed from its tiled copy) or on e4m3
    operands with per-row scales (dg_quantize_rows_e4m3 of the canvas and draw
    rows, then dg_denoise_heads_fp8); W is tiled or quantised once, when the
    object is made."""

    def __init__(self, shape, w, M, n_draw, fp8=False, device="cuda"):
        f32, i32, u8, bf = torch.float32, torch.int32, torch.uint8, torch.bfloat16
        V, D = shape.V, shape.D
        self.shape, self.M, self.n_draw, self.fp8 = shape, M, n_draw, fp8
        self.dims = dg.make_dims(d_model=D, V=V)
        nd = max(n_draw, 1)
        self.h = torch.empty((M, D), dtype=bf, device=device)
        self.draw_rows = torch.empty((nd, D), dtype=bf, device=device)
        self.inv_t = torch.empty(M, dtype=f32, device=device)
        self.inv_t_draw = torch.empty(nd, dtype=f32, device=device)
        self.lse, self.ent, self.maxz, self.prob_scale = (torch.empty(M, dtype=f32, device=device)
                                                          for _ in range(4))
        self.argmax = torch.empty(M, dtype=i32, device=device)
        self.lse_draw = torch.empty(nd, dtype=f32, device=device)
        self.probs_ld = dg.dg_probs_ld(V)
        self.probs = torch.empty((M, self.probs_ld), dtype=bf, device=device)
        self.ws = torch.empty(dg.dg_workspace_bytes(self.dims, dg.DG_WS_HEADS, M), dtype=u8,
                              device=device)
        self.w, self.w_tiled = w, None
        if fp8:
            self.w8 = torch.empty((V, D), dtype=u8, device=device)
            self.w_scale = torch.empty(V, dtype=f32, device=device)
            dg._check(dg.dg_quantize_rows_e4m3(w, V, D, self.w8, self.w_scale),
                      "dg_quantize_rows_e4m3")
            self.h8 = torch.empty((M, D), dtype=u8, device=device)
            self.h_scale = torch.empty(M, dtype=f32, device=device)
            self.d8 = torch.empty((nd, D), dtype=u8, device=device)
            self.d_scale = torch.empty(nd, dtype=f32, device=device)
        elif n_draw and dg.dg_heads_weights_bytes(self.dims):
            self.w_tiled = torch.empty(dg.dg_heads_weights_bytes(self.dims) // 2, dtype=bf,
                                       device=device)
            dg._check(dg.dg_heads_weights_tile(self.dims, w, self.w_tiled),
                      "dg_heads_weights_tile")

    def run(self, step_idx=0, stream=None):
        """Enqueue one pass; returns the number of library kernels."""
        d, nd = self.dims, self.n_draw
        if not self.fp8:
            dg._check(dg.dg_denoise_heads(d, self.h, self.M, self.draw_rows if nd else None, nd,
                                          self.w, self.inv_t, self.inv_t_draw, self.lse,
                                          self.ent, self.maxz, self.argmax, self.lse_draw,
                                          None, None, 0, None, self.prob_scale, self.probs,
                                          self.probs_ld, self.ws, stream, w_tiled=self.w_tiled),
                      "dg_denoise_heads")
            return 3
        D = self.shape.D
        dg._check(dg.dg_quantize_rows_e4m3(self.h, self.M, D, self.h8, self.h_scale, stream),
                  "dg_quantize_rows_e4m3")
        if nd:
            dg._check(dg.dg_quantize_rows_e4m3(self.draw_rows, nd, D, self.d8, self.d_scale,
                                               stream), "dg_quantize_rows_e4m3")
        dg._check(dg.dg_denoise_heads_fp8(d, self.h8, self.h_scale, self.M,
                                          self.d8 if nd else None, self.d_scale if nd else None,
                                          nd, self.w8, self.w_scale, self.inv_t, self.inv_t_draw,
                                          self.lse, self.ent, self.maxz, self.argmax,
                                          self.lse_draw, None, None, 0, None, self.prob_scale,
                                          self.probs, self.probs_ld, self.ws, stream),
                  "dg_denoise_heads_fp8")
        return 3 + (2 if nd else 1)


class SelfCond:
    """The expected-embedding GEMM of self-conditioning from given probabilities
    (dg_denoise_heads' output layout: P~ [M, probs_ld] bf16 and prob_scale = 1/S),
    on bf16 operands (dg_selfcond_from_probs) or on e4m3 operands
    (dg_quantize_rows_e4m3 of the probabilities, then dg_selfcond_from_probs8; E
    is quantised per d_model column and transposed once, when the object is made,
    by dg_quantize_cols_e4m3)."""

    def __init__(self, shape, e, M, fp8=False, device="cuda"):
        f32, u8 = torch.float32, torch.uint8
        V, D = shape.V, shape.D
        self.shape, self.M, self.fp8 = shape, M, fp8
        self.dims = dg.make_dims(d_model=D, V=V)
        self.probs_ld = dg.dg_probs_ld(V)
        self.probs = torch.empty((M, self.probs_ld), dtype=torch.bfloat16, device=device)
        self.prob_scale = torch.empty(M, dtype=f32, device=device)
        self.out = torch.empty((M, D), dtype=f32, device=device)
        self.e = e
        which = dg.DG_WS_PROBS_EMBED8 if fp8 else dg.DG_WS_PROBS_EMBED
        self.ws = torch.empty(dg.dg_workspace_bytes(self.dims, which, M), dtype=u8, device=device)
        if fp8:
            if self.probs_ld != V:
                raise ValueError("the 8-bit path quantises whole probability rows: V % 64 == 0")
            self.e8t = torch.empty((D, V), dtype=u8, device=device)
            self.e_scale = torch.empty(D, dtype=f32, device=device)
            dg._check(dg.dg_quantize_cols_e4m3(e, V, D, self.e8t, self.e_scale),
                      "dg_quantize_cols_e4m3")
            self.p8 = torch.empty((M, V), dtype=u8, device=device)
            self.p_scale = torch.empty(M, dtype=f32, device=device)

    def run(self, step_idx=0, stream=None):
        """Enqueue one pass; returns the number of library kernels."""
        d, M, V = self.dims, self.M, self.shape.V
        if not self.fp8:
            dg._check(dg.dg_selfcond_from_probs(d, self.probs, self.probs_ld, self.prob_scale, M,
                                                self.e, self.out, self.ws, stream),
                      "dg_selfcond_from_probs")
            return 2
        dg._check(dg.dg_quantize_rows_e4m3(self.probs, M, V, self.p8, self.p_scale, stream),
                  "dg_quantize_rows_e4m3")
        dg._check(dg.dg_selfcond_from_probs8(d, self.p8, self.p_scale, self.prob_scale, M,
                                             self.e8t, self.e_scale, self.out, self.ws, stream),
                  "dg_selfcond_from_probs8")
        return (3 if V >= 16384 else 1) + 2


class MixedAttention:
    """One attention launch over decoder-mode requests (canvas rows over their prompt KV)
    and encoder-mode requests (causal over their prompt rows), dg_attn_mixed."""

    def __init__(self, mode, rows, prompt_len, C, Hq, Hkv, d_head, W, device="cuda"):
        bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8
        B = len(mode)
        P = max(max(prompt_len), 1)
        self.B, self.C = B, C
        self.dims = dg.make_dims(B=B, C=C, P_max=P, Hq=Hq, Hkv=Hkv, d_head=d_head, W=W)
        self.mode = _dev(mode, i32, device)
        self.rows = _dev(rows, i32, device)
        self.prompt_len = _dev(prompt_len, i32, device)
        self.rows_host, self.mode_host, self.plen_host = list(rows), list(mode), list(prompt_len)
        self.q = torch.empty((B, C, Hq, d_head), dtype=bf, device=device)
        self.kc = torch.empty((B, C, Hkv, d_head), dtype=bf, device=device)
        self.vc = torch.empty_like(self.kc)
        self.kenc = torch.empty((B, P, Hkv, d_head), dtype=bf, device=device)
        self.venc = torch.empty_like(self.kenc)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((B, Hq, C), dtype=f32, device=device)
        self.ws = torch.empty(max(dg.dg_workspace_bytes(self.dims, dg.DG_WS_ATTN, 0), 256),
                              dtype=u8, device=device)

    def run(self, step_idx=0, stream=None):
        """Enqueue the launch; returns the number of library kernels."""
        dg._check(dg.dg_attn_mixed(self.dims, self.mode, self.rows, self.q, self.kc, self.vc,
                                   self.kenc, self.venc, None, 0, 0, 0, self.prompt_len, self.out,
                                   self.lse, self.ws, stream), "dg_attn_mixed")
        return 1 if dg.dg_workspace_bytes(self.dims, dg.DG_WS_ATTN, 0) <= 256 else 2
