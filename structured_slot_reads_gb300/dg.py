"""ctypes binding of libdg: the same call names as include/dg.h, marshalling only.

Tensor arguments may be torch tensors (their data_ptr is passed), raw integer
addresses, or None (NULL).  ``stream`` defaults to torch's current CUDA stream.
Every compute step runs in the library's CUDA kernels; loading fails loudly if
the in-tree library has not been built.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdg.so")

DG_OK = 0
DG_ERR_ARG = -1
DG_ERR_TOO_MANY_LABELS = -2
DG_ERR_LABEL = -3
DG_ERR_SHAPE = -4
DG_ERR_CUDA = -5
DG_ERR_WORKSPACE = -6
DG_DEV_TIMEOUT, DG_DEV_BAD_PAGE, DG_DEV_BAD_LABEL, DG_DEV_BAD_INDEX = 1, 2, 4, 8
DG_DEV_RANGE = 16
DG_WS_ATTN, DG_WS_LMHEAD, DG_WS_SLOT_READ, DG_WS_SELFCOND = 1, 2, 3, 4
DG_WS_HEADS, DG_WS_PROBS_EMBED, DG_WS_PREFILL, DG_WS_PROBS_EMBED8 = 5, 6, 7, 8
DG_WS_LMHEAD_NVFP4_MMA = 9
DG_MAX_LABELS = MAX_LABELS = 26
DG_MAX_WIDE_LABELS = 256
DG_NOALLOC_MAX_ROWS = 512


class DgError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "C", "P_max", "Hq", "Hkv", "d_head", "W", "d_model", "V", "sm_share")]


def make_dims(B=1, C=1, P_max=0, Hq=1, Hkv=1, d_head=64, W=0, d_model=8, V=8, sm_share=0):
    return Dims(B, C, P_max, Hq, Hkv, d_head, W, d_model, V, sm_share)


def dims_of(shape, sm_share=0):
    """Dims from a configs.StepShape."""
    return Dims(shape.B, shape.C, shape.P, shape.Hq, shape.Hkv, shape.d_head, shape.W,
                shape.D, shape.V, sm_share)


_lib = None
P, I, Z, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64, ctypes.c_float
DP = ctypes.POINTER(Dims)

_SIGS = {
    "dg_attn_decode": [DP, P, P, P, P, P, P, I, I, I, P, P, P, P, Z, P],
    "dg_lmhead_logsoftmax_entropy": [DP, P, I, P, P, P, P, P, I, P, P, P, P, P, P, Z, P],
    "dg_slot_noise": [DP, P, I, P, P, P, P, I, I, U64, I, P, P, P, P],
    "dg_slot_finish": [DP, P, P, P, P, P, P, I, I, I, F, P, P, P, P, P, P, P],
    "dg_slot_read": [DP, P, I, P, P, P, P, P, P, P, I, U64, I, I, F, P, P, P, P, P, P, P, P, Z,
                     P],
    "dg_slot_read_wide": [DP, P, I, P, P, P, P, P, P, P, I, I, U64, I, I, F, P, P, P, P, P, P, P,
                          P, Z, P],
    "dg_prefill_attn": [DP, P, P, P, P, P, P, P, I, I, I, P, P, P, Z, P],
    "dg_attn_mixed": [DP, P, P, P, P, P, P, P, P, I, I, I, P, P, P, P, Z, P],
    "dg_check_wait_timeout": [ctypes.c_int64, P, P],
    "dg_quantize_rows_e4m3": [P, I, I, P, P, P],
    "dg_quantize_cols_e4m3": [P, I, I, P, P, P],
    "dg_selfcond_from_probs8": [DP, P, P, P, I, P, P, P, P, Z, P],
    "dg_lmhead_logsoftmax_entropy_fp8": [DP, P, P, I, P, P, P, P, P, P, I, P, P, P, P, P, P, Z,
                                         P],
    "dg_quantize_nvfp4": [P, I, I, P, P, P, P],
    "dg_lmhead_logsoftmax_entropy_nvfp4": [DP, P, I, P, P, P, P, P, P, P, I, P, P, P, P, P, P,
                                           Z, P],
    "dg_quantize_nvfp4_mma": [P, I, I, P, P, P, P],
    "dg_nvfp4_mma_codes_bytes": [I, I],
    "dg_lmhead_logsoftmax_entropy_nvfp4_mma": [DP, P, I, P, P, P, P, P, P, P, I, P, P, P, P, P,
                                               P, Z, P],
    "dg_commit": [DP, P, P, P, P, P, P, P, P, P, P],
    "dg_selfcond_embed": [DP, P, I, P, P, P, P, P, P, Z, P],
    "dg_denoise_heads": [DP, P, I, P, I, P, P, P, P, P, P, P, P, P, P, P, I, P, P, P, Z, P, Z, P],
    "dg_denoise_heads_fp8": [DP, P, P, I, P, P, I, P, P, P, P, P, P, P, P, P, P, P, I, P, P, P,
                             Z, P, Z, P],
    "dg_heads_weights_bytes": [DP],
    "dg_heads_weights_tile": [DP, P, P, P],
    "dg_selfcond_from_probs": [DP, P, Z, P, I, P, P, P, Z, P],
    "dg_probs_ld": [I],
    "dg_ask_if_select": [P, I, P, P, P, P, P, I, I, P, P, P, P],
    "dg_lmhead_logsoftmax_entropy_noalloc": [DP, P, I, P, P, P, P, P, P, P],
    "dg_canvas_update": [DP, P, P, P, P, P, I, P, P],
    "dg_philox_fill": [U64, P, I, P, P],
    "dg_validate_slots": [DP, P, P, P, I, I],
    "dg_validate_slots_wide": [DP, P, P, P, I, I, I],
    "dg_workspace_bytes": [DP, I, I],
    "dg_get_status": [P, P],
    "dg_clear_status": [P],
    "dg_strerror": [I],
    "dg_num_sms": [],
}
_RES = {"dg_workspace_bytes": Z, "dg_strerror": ctypes.c_char_p, "dg_probs_ld": Z,
        "dg_heads_weights_bytes": Z, "dg_nvfp4_mma_codes_bytes": Z}


def lib():
    """Load libdg.so (once).  Raises if the library has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdg.so not built at {LIB_PATH}; run "
                               "python -m structured_slot_reads_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RES.get(name, ctypes.c_int)
        _lib = L
    return _lib


def strerror(code):
    return lib().dg_strerror(int(code)).decode()


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


def _check(code, what):
    if code != DG_OK:
        raise DgError(code, what)
    return code


# ---- the entry points, same names and argument order as include/dg.h -------
def dg_attn_decode(dims, q, kc, vc, kenc, venc, page_table, pages_per_req, n_pages, page_size,
                   prompt_len, out, lse, workspace, stream=None):
    return lib().dg_attn_decode(ctypes.byref(dims), _p(q), _p(kc), _p(vc), _p(kenc), _p(venc),
                                _p(page_table), pages_per_req, n_pages, page_size,
                                _p(prompt_len), _p(out), _p(lse), _p(workspace),
                                _nbytes(workspace), _s(stream))


def dg_lmhead_logsoftmax_entropy(dims, h, M, w, inv_t, slot_row, label_ids, n_labels, S, lse,
                                 entropy, maxz, argmax, label_lp, workspace, stream=None):
    return lib().dg_lmhead_logsoftmax_entropy(ctypes.byref(dims), _p(h), M, _p(w), _p(inv_t),
                                              _p(slot_row), _p(label_ids), _p(n_labels), S,
                                              _p(lse), _p(entropy), _p(maxz), _p(argmax),
                                              _p(label_lp), _p(workspace), _nbytes(workspace),
                                              _s(stream))


def dg_slot_noise(dims, h, M, e, inv_t, slot_row, slot_req, S, R, seed, step, rows_out,
                  inv_t_out, noise_tok_out=None, stream=None):
    return lib().dg_slot_noise(ctypes.byref(dims), _p(h), M, _p(e), _p(inv_t), _p(slot_row),
                               _p(slot_req), S, R, seed, step, _p(rows_out), _p(inv_t_out),
                               _p(noise_tok_out), _s(stream))


def dg_slot_finish(dims, rows, inv_t_rows, lse_rows, w, label_ids, n_labels, S, R, samples,
                   gate, q_avg, h_slot, chosen, lp_draws, resampled, n_reads, stream=None):
    return lib().dg_slot_finish(ctypes.byref(dims), _p(rows), _p(inv_t_rows), _p(lse_rows), _p(w),
                                _p(label_ids), _p(n_labels), S, R, samples, gate, _p(q_avg),
                                _p(h_slot), _p(chosen), _p(lp_draws), _p(resampled),
                                _p(n_reads), _s(stream))


def dg_slot_read(dims, h, M, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, S, seed, step,
                 samples, gate, q_avg, h_slot, chosen, lp_draws, resampled, n_reads,
                 noise_tok_out, workspace, stream=None):
    return lib().dg_slot_read(ctypes.byref(dims), _p(h), M, _p(w), _p(e), _p(inv_t),
                              _p(slot_row), _p(slot_req), _p(label_ids), _p(n_labels), S, seed,
                              step, samples, gate, _p(q_avg), _p(h_slot), _p(chosen),
                              _p(lp_draws), _p(resampled), _p(n_reads), _p(noise_tok_out),
                              _p(workspace), _nbytes(workspace), _s(stream))


def dg_slot_read_wide(dims, h, M, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, S, L,
                      seed, step, samples, gate, q_avg, h_slot, chosen, lp_draws, resampled,
                      n_reads, noise_tok_out, workspace, stream=None):
    return lib().dg_slot_read_wide(ctypes.byref(dims), _p(h), M, _p(w), _p(e), _p(inv_t),
                                   _p(slot_row), _p(slot_req), _p(label_ids), _p(n_labels), S, L,
                                   seed, step, samples, gate, _p(q_avg), _p(h_slot), _p(chosen),
                                   _p(lp_draws), _p(resampled), _p(n_reads), _p(noise_tok_out),
                                   _p(workspace), _nbytes(workspace), _s(stream))


def dg_prefill_attn(dims, q, k, v, prompt_len, out, lse, page_table, pages_per_req, n_pages,
                    page_size, pool_k, pool_v, workspace, stream=None):
    return lib().dg_prefill_attn(ctypes.byref(dims), _p(q), _p(k), _p(v), _p(prompt_len), _p(out),
                                 _p(lse), _p(page_table), pages_per_req, n_pages, page_size,
                                 _p(pool_k), _p(pool_v), _p(workspace), _nbytes(workspace),
                                 _s(stream))


def dg_attn_mixed(dims, mode, rows_len, q, kc, vc, kenc, venc, page_table, pages_per_req, n_pages,
                  page_size, prompt_len, out, lse, workspace, stream=None):
    return lib().dg_attn_mixed(ctypes.byref(dims), _p(mode), _p(rows_len), _p(q), _p(kc), _p(vc),
                               _p(kenc), _p(venc), _p(page_table), pages_per_req, n_pages,
                               page_size, _p(prompt_len), _p(out), _p(lse), _p(workspace),
                               _nbytes(workspace), _s(stream))


def dg_check_wait_timeout(limit_ns, waited_us, stream=None):
    return lib().dg_check_wait_timeout(int(limit_ns), _p(waited_us), _s(stream))


def dg_quantize_rows_e4m3(x, rows, cols, q, scale, stream=None):
    return lib().dg_quantize_rows_e4m3(_p(x), rows, cols, _p(q), _p(scale), _s(stream))


def dg_quantize_cols_e4m3(x, rows, cols, qt, scale, stream=None):
    return lib().dg_quantize_cols_e4m3(_p(x), rows, cols, _p(qt), _p(scale), _s(stream))


def dg_selfcond_from_probs8(dims, p8, p_scale, row_scale, M, e8t, e_scale, out, workspace,
                            stream=None):
    return lib().dg_selfcond_from_probs8(ctypes.byref(dims), _p(p8), _p(p_scale), _p(row_scale),
                                         M, _p(e8t), _p(e_scale), _p(out), _p(workspace),
                                         _nbytes(workspace), _s(stream))


def dg_lmhead_logsoftmax_entropy_fp8(dims, h8, h_scale, M, w8, w_scale, inv_t, slot_row,
                                     label_ids, n_labels, S, lse, entropy, maxz, argmax, label_lp,
                                     workspace, stream=None):
    return lib().dg_lmhead_logsoftmax_entropy_fp8(ctypes.byref(dims), _p(h8), _p(h_scale), M,
                                                  _p(w8), _p(w_scale), _p(inv_t), _p(slot_row),
                                                  _p(label_ids), _p(n_labels), S, _p(lse),
                                                  _p(entropy), _p(maxz), _p(argmax),
                                                  _p(label_lp), _p(workspace), _nbytes(workspace),
                                                  _s(stream))


def dg_quantize_nvfp4(x, rows, cols, codes, scales, g, stream=None):
    return lib().dg_quantize_nvfp4(_p(x), rows, cols, _p(codes), _p(scales), _p(g), _s(stream))


def dg_lmhead_logsoftmax_entropy_nvfp4(dims, h, M, codes, scales, g, inv_t, slot_row, label_ids,
                                       n_labels, S, lse, entropy, maxz, argmax, label_lp,
                                       workspace, stream=None):
    return lib().dg_lmhead_logsoftmax_entropy_nvfp4(ctypes.byref(dims), _p(h), M, _p(codes),
                                                    _p(scales), _p(g), _p(inv_t), _p(slot_row),
                                                    _p(label_ids), _p(n_labels), S, _p(lse),
                                                    _p(entropy), _p(maxz), _p(argmax),
                                                    _p(label_lp), _p(workspace),
                                                    _nbytes(workspace), _s(stream))


def dg_nvfp4_mma_codes_bytes(rows, cols):
    return lib().dg_nvfp4_mma_codes_bytes(rows, cols)


def dg_quantize_nvfp4_mma(x, rows, cols, codes, sf, g, stream=None):
    return lib().dg_quantize_nvfp4_mma(_p(x), rows, cols, _p(codes), _p(sf), _p(g), _s(stream))


def dg_lmhead_logsoftmax_entropy_nvfp4_mma(dims, h, M, codes, sf, g, inv_t, slot_row, label_ids,
                                           n_labels, S, lse, entropy, maxz, argmax, label_lp,
                                           workspace, stream=None):
    return lib().dg_lmhead_logsoftmax_entropy_nvfp4_mma(ctypes.byref(dims), _p(h), M, _p(codes),
                                                        _p(sf), _p(g), _p(inv_t), _p(slot_row),
                                                        _p(label_ids), _p(n_labels), S, _p(lse),
                                                        _p(entropy), _p(maxz), _p(argmax),
                                                        _p(label_lp), _p(workspace),
                                                        _nbytes(workspace), _s(stream))


def dg_commit(dims, entropy, argmax, cand, gamma, committed_state, token_state, commit, tokens,
              n_commit, stream=None):
    return lib().dg_commit(ctypes.byref(dims), _p(entropy), _p(argmax), _p(cand), _p(gamma),
                           _p(committed_state), _p(token_state), _p(commit), _p(tokens),
                           _p(n_commit), _s(stream))


def dg_selfcond_embed(dims, h, M, w, e, inv_t, lse, out, workspace, stream=None):
    return lib().dg_selfcond_embed(ctypes.byref(dims), _p(h), M, _p(w), _p(e), _p(inv_t),
                                   _p(lse), _p(out), _p(workspace), _nbytes(workspace),
                                   _s(stream))


def dg_denoise_heads(dims, h, M, draw_rows, n_draw, w, inv_t, inv_t_draw, lse, entropy, maxz,
                     argmax, lse_draw, draw_label_ids, draw_n_labels, draw_R, draw_label_z,
                     prob_scale, probs, probs_ld, workspace, stream=None, w_tiled=None):
    return lib().dg_denoise_heads(ctypes.byref(dims), _p(h), M, _p(draw_rows), n_draw, _p(w),
                                  _p(w_tiled), _p(inv_t), _p(inv_t_draw), _p(lse), _p(entropy), _p(maxz),
                                  _p(argmax), _p(lse_draw), _p(draw_label_ids),
                                  _p(draw_n_labels), draw_R, _p(draw_label_z), _p(prob_scale),
                                  _p(probs), probs_ld, _p(workspace), _nbytes(workspace),
                                  _s(stream))


def dg_denoise_heads_fp8(dims, h8, h_scale, M, draw8, draw_scale, n_draw, w8, w_scale, inv_t,
                         inv_t_draw, lse, entropy, maxz, argmax, lse_draw, draw_label_ids,
                         draw_n_labels, draw_R, draw_label_z, prob_scale, probs, probs_ld,
                         workspace, stream=None):
    return lib().dg_denoise_heads_fp8(ctypes.byref(dims), _p(h8), _p(h_scale), M, _p(draw8),
                                      _p(draw_scale), n_draw, _p(w8), _p(w_scale), _p(inv_t),
                                      _p(inv_t_draw), _p(lse), _p(entropy), _p(maxz),
                                      _p(argmax), _p(lse_draw), _p(draw_label_ids),
                                      _p(draw_n_labels), draw_R, _p(draw_label_z),
                                      _p(prob_scale), _p(probs), probs_ld, _p(workspace),
                                      _nbytes(workspace), _s(stream))


def dg_heads_weights_bytes(dims):
    return lib().dg_heads_weights_bytes(ctypes.byref(dims))


def dg_heads_weights_tile(dims, w, w_tiled, stream=None):
    return lib().dg_heads_weights_tile(ctypes.byref(dims), _p(w), _p(w_tiled), _s(stream))


def dg_selfcond_from_probs(dims, probs, probs_ld, prob_scale, M, e, out, workspace,
                           stream=None):
    return lib().dg_selfcond_from_probs(ctypes.byref(dims), _p(probs), probs_ld, _p(prob_scale),
                                        M, _p(e), _p(out), _p(workspace), _nbytes(workspace),
                                        _s(stream))


def dg_ask_if_select(chosen1, S1, cond_slot, cond_value, q_owner, q_label_ids, q_n_labels, Q,
                     S2, label_ids2, n_labels2, fired=None, stream=None):
    return lib().dg_ask_if_select(_p(chosen1), S1, _p(cond_slot), _p(cond_value), _p(q_owner),
                                  _p(q_label_ids), _p(q_n_labels), Q, S2, _p(label_ids2),
                                  _p(n_labels2), _p(fired), _s(stream))


def dg_probs_ld(V):
    return int(lib().dg_probs_ld(V))


def dg_lmhead_logsoftmax_entropy_noalloc(dims, h, M, w, inv_t, lse, entropy, maxz, argmax,
                                         stream=None):
    """dg_lmhead_logsoftmax_entropy for callers that cannot allocate a workspace:
    the scratch is a fixed array inside the library (M <= DG_NOALLOC_MAX_ROWS)."""
    return lib().dg_lmhead_logsoftmax_entropy_noalloc(ctypes.byref(dims), _p(h), M, _p(w),
                                                      _p(inv_t), _p(lse), _p(entropy), _p(maxz),
                                                      _p(argmax), _s(stream))




def dg_canvas_update(dims, h0, e_sc, emb, tokens, committed, M, h_out, stream=None):
    return lib().dg_canvas_update(ctypes.byref(dims), _p(h0), _p(e_sc), _p(emb), _p(tokens),
                                  _p(committed), M, _p(h_out), _s(stream))


def dg_philox_fill(seed, ctr4, n, out4, stream=None):
    return lib().dg_philox_fill(seed, _p(ctr4), n, _p(out4), _s(stream))


def dg_validate_slots(dims, slot_row_host, label_ids_host, n_labels_host, S, M):
    return lib().dg_validate_slots(ctypes.byref(dims), _p(slot_row_host), _p(label_ids_host),
                                   _p(n_labels_host), S, M)


def dg_validate_slots_wide(dims, slot_row_host, label_ids_host, n_labels_host, S, L, M):
    return lib().dg_validate_slots_wide(ctypes.byref(dims), _p(slot_row_host),
                                        _p(label_ids_host), _p(n_labels_host), S, L, M)


def validate_slot_table(dims, slot_row, label_ids, n_labels, M, what="slot table"):
    """Run the library's synchronous slot-table check on host arrays (int32 copies
    are made as needed) and raise DgError if it rejects them: more labels than the
    table allows (the 26-alternative limit for 26-wide tables), a duplicate label,
    a label id outside the vocabulary or a slot row outside [0, M)."""
    import numpy as np
    row = np.ascontiguousarray(np.asarray(slot_row), dtype=np.int32)
    lab = np.ascontiguousarray(np.asarray(label_ids), dtype=np.int32)
    n = np.ascontiguousarray(np.asarray(n_labels), dtype=np.int32)
    S = int(row.shape[0])
    if S == 0:
        return
    L = int(lab.shape[1]) if lab.ndim == 2 else MAX_LABELS
    if lab.shape != (S, L) or n.shape != (S,):
        raise DgError(DG_ERR_ARG, what)
    code = (dg_validate_slots(dims, row, lab, n, S, int(M)) if L == MAX_LABELS else
            dg_validate_slots_wide(dims, row, lab, n, S, L, int(M)))
    _check(code, what)


class DgDeviceError(RuntimeError):
    """Bits of the device status word that a step found set (DG_DEV_*)."""

    NAMES = {DG_DEV_TIMEOUT: "a bounded wait timed out", DG_DEV_BAD_PAGE: "bad page index",
             DG_DEV_BAD_LABEL: "label id or count out of range",
             DG_DEV_BAD_INDEX: "slot row or token outside its tensor",
             DG_DEV_RANGE: "reserved status bit"}

    def __init__(self, status, what):
        names = [v for k, v in self.NAMES.items() if status & k]
        super().__init__(f"{what}: device status {status:#x} ({'; '.join(names)})")
        self.status = status


def check_status(stream=None, what="libdg"):
    """dg_get_status on ``stream`` (synchronises it); clears the word and raises
    DgDeviceError if any bit is set, else returns 0."""
    status = dg_get_status(stream)
    if status:
        dg_clear_status(stream)
        raise DgDeviceError(status, what)
    return 0


def dg_workspace_bytes(dims, which, rows):
    return int(lib().dg_workspace_bytes(ctypes.byref(dims), which, rows))


def dg_get_status(stream=None):
    out = ctypes.c_int32(0)
    _check(lib().dg_get_status(_s(stream), ctypes.addressof(out)), "dg_get_status")
    return out.value


def dg_clear_status(stream=None):
    return lib().dg_clear_status(_s(stream))


def dg_num_sms():
    return lib().dg_num_sms()
