"""One denoise step of the structured-read sampler on the GPU, through libdg.

``DenoiseStep`` owns the device buffers of one workload (torch allocates
them; the library never does) and enqueues the library calls of one step:

  dg_attn_decode          decoder-mode attention over prompt KV + window
  dg_slot_noise           noised slot rows of the four reads
  dg_denoise_heads        one W pass: lse / entropy / argmax of every canvas row,
                          the draw rows' lse and label logits (gathered from
                          the accumulators), bf16 probabilities for self-cond
  dg_slot_finish          renormalise over the labels, entropy gate, average
  dg_commit               entropy-ordered commit (state carried forward)
  dg_selfcond_from_probs  expected embedding softmax(z) . E from the probabilities
  dg_canvas_update        next step's canvas input rows

With more than 16 draw rows (batched requests) the slot read takes its own
pass (dg_slot_read).

In the fused path (``concurrent=True``, the default) the calls that do not
feed the self-conditioning GEMM leave the caller's stream once the heads pass
is done: the slot finish, the commit and the attention run on a side stream
while dg_selfcond_from_probs streams E (that GEMM is one wave of CTAs on
7/8 of the SMs, so they run on the SMs it leaves free; the attention plans
its grid for that eighth, ``dims.sm_share``), and the canvas update waits
for the commit.  The step is the same work either way;
``concurrent=False`` enqueues it in the order above on one stream.

``fused=False`` runs the unfused calls instead (dg_lmhead_logsoftmax_entropy,
dg_slot_read, dg_selfcond_embed), which stream W three times, on one stream.

The same object serves the end-to-end path: ``upload`` copies a step's inputs
from pinned host memory, ``download`` reads back the decisions.

Slot tables enter through ``set_slots``, which runs the library's synchronous
check on the host arrays first (sotaaz.com, "The server accepts at most 26
alternatives per question": a question with more than 26 alternatives is
refused before anything runs).  ``check`` reads the device status word after
the enqueued steps (it synchronises the stream) and raises ``dg.DgDeviceError``
if any bit is set: a wait that timed out (its kernel stopped early and left
outputs unwritten) or an index, label or page out of range.
"""
import torch

from . import dg


def as_stream(stream):
    """The torch stream of a call: the current one, a raw handle wrapped, or as given."""
    if stream is None:
        return torch.cuda.current_stream()
    if isinstance(stream, int):
        return torch.cuda.ExternalStream(stream)
    return stream


def _empty(shape, dtype, device):
    return torch.empty(tuple(shape), dtype=dtype, device=device)


class Buffers(dict):
    """Named tensors that are views of one contiguous byte buffer, ``arena``
    (256-byte aligned slices), so a whole set moves in one copy."""

    def __init__(self, arena, views):
        super().__init__(views)
        self.arena = arena


def _layout(specs):
    """Offsets of (name, shape, dtype) entries in an arena; returns (entries, bytes)."""
    off, out = 0, []
    for name, shape, dt in specs:
        n = 1
        for x in shape:
            n *= int(x)
        nb = n * torch.empty((), dtype=dt).element_size()
        out.append((name, tuple(int(x) for x in shape), dt, off, nb))
        off = (off + nb + 255) // 256 * 256
    return out, max(off, 256)


def _carve(layout, device, pin=False):
    entries, total = layout
    arena = (torch.empty(total, dtype=torch.uint8, pin_memory=True) if pin
             else torch.empty(total, dtype=torch.uint8, device=device))
    views = {name: arena[off:off + nb].view(dt).view(shape)
             for name, shape, dt, off, nb in entries}
    return Buffers(arena, views)


class DenoiseStep:
    def __init__(self, shape, w, e, device="cuda", with_slots=True, seed=0, fused=True,
                 concurrent=True):
        self.shape = shape
        self.dims = dg.dims_of(shape)
        self.device = device
        B, C, D, V = shape.B, shape.C, shape.D, shape.V
        self.M = B * C
        self.w, self.e = w, e
        bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8
        dev = device
        # per-step inputs: views of one device arena (``self.inputs``)
        dh = shape.d_head
        self.in_layout = _layout([
            ("h0", (self.M, D), bf), ("inv_t", (self.M,), f32),
            ("q", (B, C, shape.Hq, dh), bf), ("kc", (B, C, shape.Hkv, dh), bf),
            ("vc", (B, C, shape.Hkv, dh), bf), ("kenc", (B, shape.P, shape.Hkv, dh), bf),
            ("venc", (B, shape.P, shape.Hkv, dh), bf), ("cand", (B, C), u8)])
        self.inputs = _carve(self.in_layout, dev)
        for k, v in self.inputs.items():
            setattr(self, k, v)
        self.h = _empty((self.M, D), bf, dev)
        self.prompt_len = torch.full((B,), shape.P, dtype=i32, device=dev)
        self.gamma = torch.full((B,), shape.gamma, dtype=f32, device=dev)
        # outputs / state
        self.attn_out = _empty((B, C, shape.Hq, shape.d_head), bf, dev)
        self.attn_lse = _empty((B, shape.Hq, C), f32, dev)
        self.lse = _empty((self.M,), f32, dev)
        self.ent = _empty((self.M,), f32, dev)
        self.maxz = _empty((self.M,), f32, dev)
        self.argmax = _empty((self.M,), i32, dev)
        self.committed = torch.zeros((B, C), dtype=u8, device=dev)
        self.tok_state = torch.full((B, C), -1, dtype=i32, device=dev)
        self.e_sc = _empty((self.M, D), f32, dev)
        # beside the self-conditioning GEMM (which plans for 7/8 of the SMs) the
        # attention plans its grid for the SMs left over: fewer key splits
        n_sm = dg.dg_num_sms()
        self.dims_side = dg.dims_of(shape, sm_share=max(1, n_sm - n_sm * 7 // 8))
        self.ws_attn = _empty((max(dg.dg_workspace_bytes(self.dims, dg.DG_WS_ATTN, 0),
                                   dg.dg_workspace_bytes(self.dims_side, dg.DG_WS_ATTN, 0),
                                   256),), u8, dev)
        # slots (same table for every request)
        self.with_slots = with_slots and len(shape.slots) > 0
        self.seed = seed
        if self.with_slots:
            S = B * len(shape.slots)
            self.S = S
            self.slot_row = _empty((S,), i32, dev)
            self.slot_req = _empty((S,), i32, dev)
            self.label_ids = _empty((S, dg.MAX_LABELS), i32, dev)
            self.n_labels = _empty((S,), i32, dev)
            self.lp_draws = _empty((S, shape.R, dg.MAX_LABELS), f32, dev)
            self.resampled = _empty((S,), u8, dev)
            self.n_reads = _empty((S,), i32, dev)
            self.noise_tok = _empty((S, shape.R), i32, dev)
            self.ws_slot = _empty((dg.dg_workspace_bytes(self.dims, dg.DG_WS_SLOT_READ,
                                                         S * shape.R),), u8, dev)
        # the decisions read back each step: views of one device arena (``self.decisions``)
        outs = [("commit", (B, C), u8), ("tokens", (B, C), i32), ("n_commit", (B,), i32)]
        if self.with_slots:
            outs += [("q_avg", (self.S, dg.MAX_LABELS), f32), ("h_slot", (self.S,), f32),
                     ("chosen", (self.S,), i32)]
        self.out_layout = _layout(outs)
        self.decisions = _carve(self.out_layout, dev)
        for k, v in self.decisions.items():
            setattr(self, k, v)
        # fused path: one stream of W for the canvas rows, the slot draws (up to
        # 16 draw rows ride along; more go through their own dg_slot_read pass)
        # and the self-conditioning probabilities
        self.fused = fused
        self.concurrent = fused and concurrent
        self._side = None                   # side stream and its event, made on first use
        self.n_draw = self.S * shape.R if (self.with_slots and self.S * shape.R <= 16) else 0
        self.w_tiled = None
        if not self.fused:
            self.ws_lm = _empty((dg.dg_workspace_bytes(self.dims, dg.DG_WS_LMHEAD, self.M),), u8,
                                dev)
            self.ws_sc = _empty((dg.dg_workspace_bytes(self.dims, dg.DG_WS_SELFCOND, self.M),), u8,
                                dev)
        else:
            nd = max(self.n_draw, 1)
            self.draw_rows = _empty((nd, D), bf, dev)
            self.inv_t_draw = _empty((nd,), f32, dev)
            self.lse_draw = _empty((nd,), f32, dev)
            self.probs_ld = dg.dg_probs_ld(V)
            self.probs = _empty((self.M, self.probs_ld), bf, dev)
            self.prob_scale = _empty((self.M,), f32, dev)
            self.ws_heads = _empty((dg.dg_workspace_bytes(self.dims, dg.DG_WS_HEADS, self.M),), u8, dev)
            self.ws_pe = _empty((dg.dg_workspace_bytes(self.dims, dg.DG_WS_PROBS_EMBED, self.M),), u8, dev)
            # W's tiled copy, which the pass streams when the draw rows ride in it
            # (written here once; call tile_weights() again after changing w)
            if self.n_draw and dg.dg_heads_weights_bytes(self.dims):
                self.w_tiled = _empty((dg.dg_heads_weights_bytes(self.dims) // 2,), bf, dev)
                if self.w_tiled.is_cuda:
                    self.tile_weights()

    def tile_weights(self, stream=None):
        """Rewrite the tiled copy of ``w`` the heads pass streams (dg_heads_weights_tile)."""
        if self.w_tiled is not None:
            dg._check(dg.dg_heads_weights_tile(self.dims, self.w, self.w_tiled, stream),
                      "dg_heads_weights_tile")

    # ------------------------------------------------------------ slots
    def set_slots(self, slot_row, slot_req, label_ids, n_labels):
        """Load the slot table from host arrays after the library's synchronous
        check (raises dg.DgError: more than 26 labels, a duplicate or out-of-vocabulary
        label, a slot row outside the canvas rows)."""
        import numpy as np
        if not self.with_slots:
            raise ValueError("this step has no slots")
        dg.validate_slot_table(self.dims, slot_row, label_ids, n_labels, self.M)
        for name, a in (("slot_row", slot_row), ("slot_req", slot_req),
                        ("label_ids", label_ids), ("n_labels", n_labels)):
            t = torch.from_numpy(np.ascontiguousarray(np.asarray(a), dtype=np.int32))
            getattr(self, name).copy_(t.view(getattr(self, name).shape))

    def check(self, stream=None):
        """Read the device status word after the enqueued steps (synchronises
        ``stream``), clear it and raise dg.DgDeviceError if any bit was set.
        Returns 0 otherwise."""
        return dg.check_status(stream, "denoise step")

    # ------------------------------------------------------------- graphs
    def capture(self, step_idx):
        """Record step ``step_idx`` as a CUDA graph (once per step index: the noise
        draws depend on it).  Call after one eager step, so every kernel's one-time
        set-up has run; replaying the graph is the same work as ``run(step_idx)``."""
        if not hasattr(self, "_graphs"):
            self._graphs = {}
        g = self._graphs.get(step_idx)
        if g is None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.run(step_idx=step_idx)
            self._graphs[step_idx] = g
        return g

    def replay(self, step_idx):
        """Launch the captured graph of step ``step_idx``; returns the kernels it holds."""
        self.capture(step_idx).replay()
        return self.kernels_per_step()

    # ------------------------------------------------------------------ step
    def reset_state(self):
        self.committed.zero_()
        self.tok_state.fill_(-1)
        self.h.copy_(self.h0)

    def run(self, step_idx=0, stream=None):
        """Enqueue one denoise step; returns the number of library kernels launched."""
        s, d = self.shape, self.dims
        ck = dg._check
        if self.fused:
            return self._run_fused(step_idx, stream)
        self._attention(stream)
        ck(dg.dg_lmhead_logsoftmax_entropy(d, self.h, self.M, self.w, self.inv_t, None, None,
                                           None, 0, self.lse, self.ent, self.maxz, self.argmax,
                                           None, self.ws_lm, stream),
           "dg_lmhead_logsoftmax_entropy")
        if self.with_slots:
            self._slot_read(step_idx, stream)
        ck(dg.dg_commit(d, self.ent, self.argmax, self.cand, self.gamma, self.committed,
                        self.tok_state, self.commit, self.tokens, self.n_commit, stream),
           "dg_commit")
        ck(dg.dg_selfcond_embed(d, self.h, self.M, self.w, self.e, self.inv_t, self.lse,
                                self.e_sc, self.ws_sc, stream), "dg_selfcond_embed")
        ck(dg.dg_canvas_update(d, self.h0, self.e_sc, self.e, self.tok_state, self.committed,
                               self.M, self.h, stream), "dg_canvas_update")
        return self.kernels_per_step()

    def _attn_dims(self):
        """The attention's dims: on the side stream it plans for the SMs the GEMM leaves."""
        return self.dims_side if self.concurrent else self.dims

    def _attention(self, stream):
        dg._check(dg.dg_attn_decode(self._attn_dims(), self.q, self.kc, self.vc, self.kenc,
                                    self.venc, None, 0, 0, 0, self.prompt_len, self.attn_out,
                                    self.attn_lse, self.ws_attn, stream), "dg_attn_decode")

    def _selfcond(self, stream):
        dg._check(dg.dg_selfcond_from_probs(self.dims, self.probs, self.probs_ld, self.prob_scale,
                                            self.M, self.e, self.e_sc, self.ws_pe, stream),
                  "dg_selfcond_from_probs")

    def _slot_read(self, step_idx, stream):
        s, d = self.shape, self.dims
        dg._check(dg.dg_slot_read(d, self.h, self.M, self.w, self.e, self.inv_t, self.slot_row,
                                  self.slot_req, self.label_ids, self.n_labels, self.S, self.seed,
                                  step_idx, s.R, s.gate, self.q_avg, self.h_slot, self.chosen,
                                  self.lp_draws, self.resampled, self.n_reads, self.noise_tok,
                                  self.ws_slot, stream), "dg_slot_read")

    def _run_fused(self, step_idx, stream):
        s, d = self.shape, self.dims
        ck = dg._check
        main = as_stream(stream)
        if not self.concurrent:
            self._attention(main)
        if self.with_slots and not self.n_draw:
            self._slot_read(step_idx, main)
        if self.n_draw:
            ck(dg.dg_slot_noise(d, self.h, self.M, self.e, self.inv_t, self.slot_row,
                                self.slot_req, self.S, s.R, self.seed, step_idx, self.draw_rows,
                                self.inv_t_draw, self.noise_tok, main), "dg_slot_noise")
        # the draws' label logits are gathered into lp_draws by the pass
        nd = self.n_draw
        ck(dg.dg_denoise_heads(d, self.h, self.M, self.draw_rows if nd else None, nd, self.w,
                               self.inv_t, self.inv_t_draw, self.lse, self.ent, self.maxz,
                               self.argmax, self.lse_draw, self.label_ids if nd else None,
                               self.n_labels if nd else None, s.R,
                               self.lp_draws if nd else None, self.prob_scale, self.probs,
                               self.probs_ld, self.ws_heads, main, w_tiled=self.w_tiled),
           "dg_denoise_heads")
        side = main
        if self.concurrent:
            if self._side is None:
                self._side = torch.cuda.Stream(device=self.h.device), torch.cuda.Event()
            side, self.ev_commit = self._side
            # the GEMM goes first so that its CTAs are placed before the side work's
            side.wait_stream(main)
            self._selfcond(main)
        if self.n_draw:
            # the label logits came out of the heads pass (rows = None)
            ck(dg.dg_slot_finish(d, None, None, self.lse_draw, None,
                                 self.label_ids, self.n_labels, self.S, s.R, s.R, s.gate,
                                 self.q_avg, self.h_slot, self.chosen, self.lp_draws,
                                 self.resampled, self.n_reads, side), "dg_slot_finish")
        ck(dg.dg_commit(d, self.ent, self.argmax, self.cand, self.gamma, self.committed,
                        self.tok_state, self.commit, self.tokens, self.n_commit, side),
           "dg_commit")
        if self.concurrent:
            self.ev_commit.record(side)
            self._attention(side)
            main.wait_event(self.ev_commit)     # the update reads the commit's state
        else:
            self._selfcond(main)
        ck(dg.dg_canvas_update(d, self.h0, self.e_sc, self.e, self.tok_state, self.committed,
                               self.M, self.h, main), "dg_canvas_update")
        if self.concurrent:
            main.wait_stream(side)
        return self.kernels_per_step()

    def kernels_per_step(self):
        """Library kernels one step launches."""
        n = 1 + (1 if self._attn_splits() > 1 else 0)
        if self.fused:
            # ref + heads + finalize + commit + accum + reduce + update, and either
            # noise + slot epilogue with the draws in the pass (their
            # log-normalisers finalised with the canvas rows', their label logits
            # gathered by the pass), or a slot read
            n += 3 + 1 + 2 + 1
            if self.n_draw:
                n += 2
            elif self.with_slots:
                n += 4
            return n
        # stats + finalize, [noise + stats + finalize + slot epilogue], commit,
        # probs + accum + reduce, update
        n += 2
        n += 4 if self.with_slots else 0
        n += 1 + 3 + 1
        return n

    def _attn_splits(self):
        return 1 if dg.dg_workspace_bytes(self._attn_dims(), dg.DG_WS_ATTN, 0) <= 256 else 2

    # ------------------------------------------------------- host round trip
    def host_buffers(self):
        """Pinned host buffers of one step's inputs and decisions, laid out as
        the device arenas (``Buffers``: a dict of views plus ``.arena``)."""
        return _carve(self.in_layout, None, pin=True), _carve(self.out_layout, None, pin=True)

    def upload(self, ins):
        """Copy a step's inputs from host buffers; returns the bytes copied."""
        if isinstance(ins, Buffers) and ins.arena.numel() == self.inputs.arena.numel():
            self.inputs.arena.copy_(ins.arena, non_blocking=True)
            n = ins.arena.numel()
        else:
            n = 0
            for k, t in ins.items():
                getattr(self, k).copy_(t, non_blocking=True)
                n += t.numel() * t.element_size()
        self.h.copy_(self.h0)
        return n

    def download(self, outs):
        """Copy the step's decisions into host buffers; returns the bytes copied."""
        if isinstance(outs, Buffers) and outs.arena.numel() == self.decisions.arena.numel():
            outs.arena.copy_(self.decisions.arena, non_blocking=True)
            return outs.arena.numel()
        n = 0
        for k, t in outs.items():
            t.copy_(getattr(self, k), non_blocking=True)
            n += t.numel() * t.element_size()
        return n


class HostPipeline:
    """End-to-end steps with host transfers overlapped with compute.

    ``submit(step_idx, ins, outs)`` enqueues one step whose inputs come from
    the pinned host tensors ``ins`` (as from ``DenoiseStep.host_buffers``) and
    whose decisions go to the pinned host tensors ``outs``:

      upload stream    host -> staging set b (b = submission parity), once the
                       step that last read set b has finished
      compute stream   one CUDA graph of the step whose kernels read their
                       inputs from staging set b and write the decisions to
                       output staging set b (no device-side copies)
      download stream  output staging set b -> ``outs``

    So step i+1's inputs cross the link while step i computes, and step i's
    decisions come back while step i+1 computes.  Every step still makes its
    own host->device copy of all its inputs and its own device->host read of
    its decisions.  The copies are asynchronous: ``ins`` must stay unchanged
    and ``outs`` unread until ``sync()`` returns (give each in-flight step its
    own host tensors to refill them earlier).  The decisions land in ``outs``
    only (not in the step's own decision tensors); the carried state
    (committed positions, tokens, canvas rows) is the step's, as with ``run``.  Graphs are captured on first
    use, or ahead of time with ``prepare``; the step must have run once
    eagerly before (one-time set-up of its kernels).
    """

    def __init__(self, step, use_graphs=True):
        self.step = step
        self.use_graphs = use_graphs
        self.up = torch.cuda.Stream(device=step.h.device)
        self.down = torch.cuda.Stream(device=step.h.device)
        dev = step.h.device
        self.stage_in = [_carve(step.in_layout, dev) for _ in range(2)]
        self.stage_out = [_carve(step.out_layout, dev) for _ in range(2)]
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_up, self.ev_in_free, self.ev_done, self.ev_out_free = ev(), ev(), ev(), ev()
        self.graphs = {}
        self.n = 0

    def _body(self, step_idx, b):
        """The step with its inputs read from staging set b and its decisions
        written there: the input and decision tensors are bound to the staging
        arenas while the step is enqueued (or captured), then restored."""
        st = self.step
        saved = {k: getattr(st, k) for k in (*st.inputs, *st.decisions)}
        try:
            for k, v in (*self.stage_in[b].items(), *self.stage_out[b].items()):
                setattr(st, k, v)
            st.h.copy_(st.h0)
            st.run(step_idx)
        finally:
            for k, v in saved.items():
                setattr(st, k, v)

    def _graph(self, step_idx, b):
        g = self.graphs.get((step_idx, b))
        if g is None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._body(step_idx, b)
            self.graphs[(step_idx, b)] = g
        return g

    def prepare(self, step_indices):
        """Capture the graphs of the next submissions (step indices in order)."""
        for j, i in enumerate(step_indices):
            self._graph(i, (self.n + j) & 1)

    def submit(self, step_idx, ins, outs):
        """Enqueue one step; returns (host->device bytes, device->host bytes)."""
        b = self.n & 1
        main = torch.cuda.current_stream()
        with torch.cuda.stream(self.up):
            self.up.wait_event(self.ev_in_free[b])
            h2d = _copy_set(self.stage_in[b], ins)
            self.ev_up[b].record(self.up)
        main.wait_event(self.ev_up[b])
        main.wait_event(self.ev_out_free[b])
        if self.use_graphs:
            self._graph(step_idx, b).replay()
        else:
            self._body(step_idx, b)
        self.ev_in_free[b].record(main)
        self.ev_done[b].record(main)
        with torch.cuda.stream(self.down):
            self.down.wait_event(self.ev_done[b])
            d2h = _copy_set(outs, self.stage_out[b])
            self.ev_out_free[b].record(self.down)
        self.n += 1
        return h2d, d2h

    def join(self, stream=None):
        """Make ``stream`` (default: current) wait for every enqueued transfer."""
        s = stream or torch.cuda.current_stream()
        s.wait_stream(self.up)
        s.wait_stream(self.down)

    def sync(self):
        """Wait for every enqueued step and transfer, then read the device status
        word (DenoiseStep.check): raises dg.DgDeviceError if a kernel of these
        steps recorded an error (a wait that timed out, a bad label or page)."""
        self.join()
        torch.cuda.current_stream().synchronize()
        return self.step.check(torch.cuda.current_stream())


def _copy_set(dst, src):
    """Copy a set of named tensors (one copy when both are arenas of one layout);
    returns the bytes copied."""
    if isinstance(src, Buffers) and isinstance(dst, Buffers) and \
            src.arena.numel() == dst.arena.numel():
        dst.arena.copy_(src.arena, non_blocking=True)
        return src.arena.numel()
    n = 0
    for k, t in src.items():
        dst[k].copy_(t, non_blocking=True)
        n += t.numel() * t.element_size()
    return n
