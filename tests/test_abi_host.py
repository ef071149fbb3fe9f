"""Host-side checks of the C ABI (no GPU): the library loads, exports every symbol
include/dg.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

from structured_slot_reads_gb300 import dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(dg.LIB_PATH):
        from structured_slot_reads_gb300 import build
        build.build()
    return dg.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dg.h but not exported"
    assert set(names) == set(dg._SIGS), "binding and header disagree on the entry points"


def test_strerror(lib):
    assert dg.strerror(dg.DG_ERR_TOO_MANY_LABELS) == "at most 26 alternatives per slot"
    assert dg.strerror(0) == "ok"
    assert "unknown" in dg.strerror(-99)


def _slots(n_labels, ids=None, rows=None):
    S = len(n_labels)
    lab = np.full((S, 26), -1, np.int32)
    for s, n in enumerate(n_labels):
        lab[s, :min(n, 26)] = np.arange(min(n, 26)) + 10 * s if ids is None else ids[s][:min(n, 26)]
    rows = np.arange(S, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    return rows, lab, np.asarray(n_labels, np.int32)


def test_validate_slots_rejects_27_labels(lib):
    d = dg.make_dims(V=1000, d_model=8)
    rows, lab, n = _slots([2, 27])
    lab27 = np.zeros((2, 27), np.int32)  # the table is 26 wide; 27 is rejected before reading
    assert dg.dg_validate_slots(d, rows, lab, n, 2, 10) == dg.DG_ERR_TOO_MANY_LABELS


def test_validate_slots_accepts_26_and_checks_ids(lib):
    d = dg.make_dims(V=1000, d_model=8)
    rows, lab, n = _slots([2, 26, 5])
    assert dg.dg_validate_slots(d, rows, lab, n, 3, 10) == dg.DG_OK
    dup = lab.copy()
    dup[1, 3] = dup[1, 4]
    assert dg.dg_validate_slots(d, rows, dup, n, 3, 10) == dg.DG_ERR_LABEL
    big = lab.copy()
    big[2, 0] = 1000
    assert dg.dg_validate_slots(d, rows, big, n, 3, 10) == dg.DG_ERR_LABEL
    assert dg.dg_validate_slots(d, np.array([0, 1, 10], np.int32), lab, n, 3, 10) == dg.DG_ERR_SHAPE
    assert dg.dg_validate_slots(d, rows, lab, np.array([2, 0, 5], np.int32), 3, 10) == dg.DG_ERR_LABEL


def test_workspace_sizes(lib):
    from structured_slot_reads_gb300 import configs
    for shp in configs.ALL.values():
        d = dg.dims_of(shp)
        assert dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, shp.B * shp.C) > 0
        assert dg.dg_workspace_bytes(d, dg.DG_WS_SELFCOND, shp.B * shp.C) >= shp.B * shp.C * shp.V * 2
        assert dg.dg_workspace_bytes(d, dg.DG_WS_ATTN, 0) > 0
        assert dg.dg_workspace_bytes(d, dg.DG_WS_SLOT_READ, 12) > 12 * shp.D * 2
    bad = dg.make_dims(d_model=12)
    assert dg.dg_workspace_bytes(bad, dg.DG_WS_LMHEAD, 4) == 0
    assert dg.dg_workspace_bytes(dg.make_dims(Hq=3, Hkv=2), dg.DG_WS_ATTN, 0) == 0
    assert dg.dg_workspace_bytes(dg.make_dims(), 99, 1) == 0


def test_compute_calls_validate_before_launch(lib):
    d = dg.make_dims(B=1, C=32, P_max=64, Hq=2, Hkv=1, d_head=64, W=8, d_model=128, V=1024)
    # null pointers
    assert dg.dg_lmhead_logsoftmax_entropy(d, None, 4, None, None, None, None, None, 0, None,
                                           None, None, None, None, None,
                                           stream=0) == dg.DG_ERR_ARG
    assert dg.dg_attn_decode(d, None, None, None, None, None, None, 0, 0, 0, None, None, None,
                             None, stream=0) == dg.DG_ERR_ARG
    assert dg.dg_commit(d, None, None, None, None, None, None, None, None, None,
                        stream=0) == dg.DG_ERR_ARG
    # unsupported shapes
    bad = dg.make_dims(B=1, C=32, P_max=64, Hq=2, Hkv=1, d_head=128, W=8, d_model=128, V=1024)
    assert dg.dg_attn_decode(bad, 16, 16, 16, 16, 16, None, 0, 0, 0, 16, 16, 16, None,
                             stream=0) == dg.DG_ERR_SHAPE
    gqa = dg.make_dims(B=1, C=32, P_max=64, Hq=3, Hkv=2, d_head=64, W=8, d_model=128, V=1024)
    assert dg.dg_attn_decode(gqa, 16, 16, 16, 16, 16, None, 0, 0, 0, 16, 16, 16, None,
                             stream=0) == dg.DG_ERR_SHAPE
    assert dg.dg_commit(dg.make_dims(B=1, C=2000), 16, 16, 16, 16, None, None, 16, 16, 16,
                        stream=0) == dg.DG_ERR_SHAPE
    # misaligned TMA operand
    assert dg.dg_lmhead_logsoftmax_entropy(d, 18, 4, 16, 16, None, None, None, 0, 16, 16, 16,
                                           16, None, None, stream=0) == dg.DG_ERR_ARG
    # non power-of-two vocabulary for the noise map
    d1000 = dg.make_dims(d_model=128, V=1000)
    assert dg.dg_slot_noise(d1000, 16, 4, 16, 16, 16, 16, 1, 4, 0, 0, 16, 16, None,
                            stream=0) == dg.DG_ERR_SHAPE
    # samples outside [1, R]
    assert dg.dg_slot_finish(d, 16, 16, 16, 16, 16, 16, 1, 4, 5, 0.1, 16, 16, 16, 16, 16, 16,
                             stream=0) == dg.DG_ERR_ARG
    # workspace missing
    assert dg.dg_lmhead_logsoftmax_entropy(d, 16, 4, 16, 16, None, None, None, 0, 16, 16, 16,
                                           16, None, None, stream=0) == dg.DG_ERR_WORKSPACE
    # a label gather: negative slot count, a missing slot table
    assert dg.dg_lmhead_logsoftmax_entropy(d, 16, 4, 16, 16, None, None, None, -1, 16, 16, 16,
                                           16, None, None, stream=0) == dg.DG_ERR_ARG


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(dg, "_lib", None)
    monkeypatch.setattr(dg, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dg.lib()


def test_binding_constants_match_header():
    text = open(HEADER).read()
    defs = re.findall(r"#define\s+(DG_[A-Z0-9_]+)\s+\(?(-?\d+)\)?", text)
    assert len(defs) >= 18
    for name, val in defs:
        assert hasattr(dg, name), f"{name} missing from the binding"
        assert getattr(dg, name) == int(val), f"{name}: binding {getattr(dg, name)} != header {val}"


def test_binding_dims_match_header():
    """dg_dims in the header and the binding's ctypes structure: same int fields, same order."""
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} dg_dims;", text, re.S).group(1)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            assert decl.startswith("int "), decl
            fields += [f.strip() for f in decl[4:].split(",")]
    assert [f for f, _ in dg.Dims._fields_] == fields
    assert all(t is ctypes.c_int for _, t in dg.Dims._fields_)
    assert ctypes.sizeof(dg.Dims) == 4 * len(fields)
    assert dg.make_dims().sm_share == 0 and dg.make_dims(sm_share=19).sm_share == 19


@pytest.mark.parametrize("fused", [True, False])
def test_step_runner_builds_on_host(lib, fused):
    """The step runner's set-up uses only host-side library calls (workspace sizes)."""
    import torch

    from structured_slot_reads_gb300 import configs
    from structured_slot_reads_gb300.step import DenoiseStep
    shp = configs.TINY
    w = torch.zeros((shp.V, shp.D), dtype=torch.bfloat16)
    st = DenoiseStep(shp, w, w, device="cpu", fused=fused)
    assert st.fused == fused
    assert st.kernels_per_step() == (11 if fused else 13) - (0 if st._attn_splits() > 1 else 1)
    if fused:
        assert st.probs.shape == (shp.C, dg.dg_probs_ld(shp.V)) and st.n_draw == 4
        # the pass streams W from its tiled copy (whole 224-row tiles)
        assert st.w_tiled.numel() * 2 == dg.dg_heads_weights_bytes(st.dims)
        assert st.w_tiled.numel() == -(-shp.V // 224) * 224 * shp.D


def test_batched_step_reads_slots_in_their_own_pass(lib):
    """With more than 16 draw rows the fused step reads the slots through dg_slot_read."""
    import torch

    from structured_slot_reads_gb300 import configs
    from structured_slot_reads_gb300.step import DenoiseStep
    shp = configs.scaled(configs.TINY, B=8)
    w = torch.zeros((shp.V, shp.D), dtype=torch.bfloat16)
    st = DenoiseStep(shp, w, w, device="cpu", fused=True)
    assert st.S == 8 and st.n_draw == 0 and not hasattr(st, "ws_sc") and st.w_tiled is None
    assert st.kernels_per_step() == 13 - (0 if st._attn_splits() > 1 else 1)


def test_two_stage_runner_builds_on_host(lib):
    """The batched two-stage runner sets up its tables with host-side calls only, and
    its page table covers the longest prompt (the attention call's shape check)."""
    import torch

    from structured_slot_reads_gb300 import configs, inputs
    from structured_slot_reads_gb300.read import TwoStageRead
    shp = configs.scaled(configs.MIXED_BATCH, B=4, C=64, P=200, D=256, V=4096)
    tables = inputs.two_stage_tables(shp, 3)
    plen = inputs.prompt_lengths(shp, 3, lo=100)
    w = torch.zeros((shp.V, shp.D), dtype=torch.bfloat16)
    tr = TwoStageRead(shp, w, w, tables, plen, device="cpu", seed=3)
    assert tr.S1 == sum(1 + len(t["others"]) for t in tables)
    assert tr.Q == shp.B * 9 and tr.S2 == shp.B
    assert tr.pages_per_req * shp.page_size >= tr.dims.P_max == int(plen.max())
    assert all(tr.host_slots1[0][g] // shp.C == b for b, g in enumerate(tr.group_slot))
    assert dg.dg_ask_if_select(None, 1, None, None, None, None, None, 2, 1, 16, 16,
                               stream=0) == dg.DG_ERR_ARG
    assert dg.dg_ask_if_select(16, 1, 16, 16, 16, 16, 16, 2, -1, 16, 16,
                               stream=0) == dg.DG_ERR_ARG


def test_wide_read_rejects_tables_wider_than_256(lib):
    d = dg.make_dims(d_model=128, V=1024)
    rc = dg.dg_slot_read_wide(d, 16, 4, 16, 16, 16, 16, 16, 16, 16, 1, 257, 0, 0, 4, 0.1, 16, 16,
                              16, 16, 16, 16, None, None, stream=0)
    assert rc == dg.DG_ERR_TOO_MANY_LABELS
    rc = dg.dg_slot_read_wide(d, 16, 4, 16, 16, 16, 16, 16, 16, 16, 1, 0, 0, 0, 4, 0.1, 16, 16,
                              16, 16, 16, 16, None, None, stream=0)
    assert rc == dg.DG_ERR_TOO_MANY_LABELS


def test_prefill_validates_shapes(lib):
    ok = dg.make_dims(B=1, P_max=64, Hq=8, Hkv=2, d_head=512)
    assert dg.dg_workspace_bytes(ok, dg.DG_WS_PREFILL, 0) > 0
    bad_d = dg.make_dims(B=1, P_max=64, Hq=8, Hkv=2, d_head=64)
    assert dg.dg_prefill_attn(bad_d, 16, 16, 16, 16, 16, 16, None, 0, 0, 0, None, None, None,
                              stream=0) == dg.DG_ERR_SHAPE
    assert dg.dg_prefill_attn(ok, None, 16, 16, 16, 16, 16, None, 0, 0, 0, None, None, None,
                              stream=0) == dg.DG_ERR_ARG
    assert dg.dg_prefill_attn(ok, 16, 16, 16, 16, 16, 16, None, 0, 0, 0, None, None, None,
                              stream=0) == dg.DG_ERR_WORKSPACE


def test_mixed_attention_validates(lib):
    d = dg.make_dims(B=2, C=64, P_max=32, Hq=8, Hkv=2, d_head=512, W=8)
    assert dg.dg_attn_mixed(d, None, 16, 16, 16, 16, 16, 16, None, 0, 0, 0, 16, 16, 16, None,
                            stream=0) == dg.DG_ERR_ARG
    d64 = dg.make_dims(B=2, C=64, P_max=32, Hq=8, Hkv=2, d_head=64, W=8)
    assert dg.dg_attn_mixed(d64, 16, 16, 16, 16, 16, 16, 16, None, 0, 0, 0, 16, 16, 16, None,
                            stream=0) == dg.DG_ERR_SHAPE
    assert dg.dg_attn_mixed(d, 16, 16, 16, 16, 16, 16, 16, 16, 2, 10, 24, 16, 16, 16, None,
                            stream=0) == dg.DG_ERR_SHAPE   # 24-key pages: not on this kernel


def test_wait_timeout_diagnostic_validates_its_limit(lib):
    assert dg.dg_check_wait_timeout(0, 16, stream=0) == dg.DG_ERR_ARG
    assert dg.dg_check_wait_timeout(2_000_000_000, 16, stream=0) == dg.DG_ERR_ARG
    assert dg.dg_check_wait_timeout(1000, None, stream=0) == dg.DG_ERR_ARG


def test_heads_pass_wants_32_byte_aligned_probabilities(lib):
    """The probabilities are written with 256-bit stores."""
    d = dg.make_dims(d_model=128, V=1024)
    ld = dg.dg_probs_ld(1024)
    args = lambda probs: (d, 32, 4, None, 0, 32, 32, None, 32, 32, 32, 32, None,  # noqa: E731
                          None, None, 0, None, 32, probs, ld, None)
    assert dg.dg_denoise_heads(*args(48), stream=0) == dg.DG_ERR_ARG        # 16- not 32-aligned
    assert dg.dg_denoise_heads(*args(64), stream=0) == dg.DG_ERR_WORKSPACE  # alignment accepted


def test_heads_weights_tiled_copy_validates(lib):
    """The tiled copy of W: ceil(V / 224) whole tiles of d_model columns, only for
    d_model a multiple of 64; refusals come before any launch."""
    d = dg.make_dims(d_model=2816, V=262144)
    assert dg.dg_heads_weights_bytes(d) == 1171 * 224 * 2816 * 2
    assert dg.dg_heads_weights_bytes(dg.make_dims(d_model=128, V=224)) == 224 * 128 * 2
    assert dg.dg_heads_weights_bytes(dg.make_dims(d_model=128, V=225)) == 2 * 224 * 128 * 2
    d96 = dg.make_dims(d_model=96, V=1024)
    assert dg.dg_heads_weights_bytes(d96) == 0
    assert dg.dg_heads_weights_tile(d96, 32, 32, stream=0) == dg.DG_ERR_SHAPE
    d128 = dg.make_dims(d_model=128, V=1024)
    assert dg.dg_heads_weights_tile(d128, None, 32, stream=0) == dg.DG_ERR_ARG
    assert dg.dg_heads_weights_tile(d128, 32, 40, stream=0) == dg.DG_ERR_ARG   # 8-byte aligned
    # the pass refuses a tiled copy it cannot use (d_model not a multiple of 64)
    ld = dg.dg_probs_ld(1024)
    args = (d96, 32, 4, None, 0, 32, 32, None, 32, 32, 32, 32, None, None, None, 0, None, 32,
            64, ld, None)
    assert dg.dg_denoise_heads(*args, stream=0, w_tiled=32) == dg.DG_ERR_ARG
    assert dg.dg_denoise_heads(*args, stream=0) == dg.DG_ERR_WORKSPACE


def test_fp8_heads_pass_validates(lib):
    """dg_denoise_heads_fp8 refuses before any launch: d_model not a multiple of 16,
    more than 16 draw rows, a W-scale vector not 16-byte aligned, a missing
    workspace."""
    d = dg.make_dims(d_model=128, V=1024)
    ld = dg.dg_probs_ld(1024)

    def call(dims=d, n_draw=0, w_scale=64, ws=None):
        return dg.dg_denoise_heads_fp8(dims, 64, 64, 4, 64 if n_draw else None,
                                       64 if n_draw else None, n_draw, 64, w_scale, 64,
                                       64 if n_draw else None, 64, 64, 64, 64,
                                       64 if n_draw else None, None, None, 0, None, 64, 64, ld,
                                       ws, stream=0)
    assert call(dims=dg.make_dims(d_model=120, V=1024)) == dg.DG_ERR_SHAPE
    assert call(n_draw=17) == dg.DG_ERR_ARG
    assert call(w_scale=72) == dg.DG_ERR_ARG          # 8-byte aligned
    assert call() == dg.DG_ERR_WORKSPACE              # everything else accepted


def test_8bit_self_conditioning_validates(lib):
    d = dg.make_dims(d_model=128, V=1024)
    ok = (d, 32, 32, None, 4, 32, 32, 32, None)
    assert dg.dg_selfcond_from_probs8(*ok, stream=0) == dg.DG_ERR_WORKSPACE
    assert dg.dg_selfcond_from_probs8(dg.make_dims(d_model=128, V=1000), *ok[1:],
                                      stream=0) == dg.DG_ERR_SHAPE          # V % 16
    assert dg.dg_selfcond_from_probs8(dg.make_dims(d_model=126, V=1024), *ok[1:],
                                      stream=0) == dg.DG_ERR_SHAPE          # d_model % 4
    assert dg.dg_selfcond_from_probs8(d, 40, 32, None, 4, 32, 32, 32, None,
                                      stream=0) == dg.DG_ERR_ARG            # p8 not 16-aligned
    assert dg.dg_selfcond_from_probs8(d, None, 32, None, 4, 32, 32, 32, None,
                                      stream=0) == dg.DG_ERR_ARG
    assert dg.dg_quantize_cols_e4m3(None, -1, 4, None, None, stream=0) == dg.DG_ERR_ARG
    assert dg.dg_quantize_cols_e4m3(None, 4, 4, None, None, stream=0) == dg.DG_ERR_ARG
    assert dg.dg_quantize_cols_e4m3(None, 0, 4, None, None, stream=0) == dg.DG_OK


def test_validate_slots_wide(lib):
    """Tables of stride L for the wide read: up to L labels per slot, L <= 256."""
    d = dg.make_dims(V=5000, d_model=8)
    lab = np.full((2, 77), -1, np.int32)
    lab[0, :77] = np.arange(77)
    lab[1, :3] = [7, 8, 9]
    n = np.array([77, 3], np.int32)
    rows = np.array([0, 5], np.int32)
    assert dg.dg_validate_slots_wide(d, rows, lab, n, 2, 77, 10) == dg.DG_OK
    assert dg.dg_validate_slots_wide(d, rows, lab, np.array([78, 3], np.int32), 2, 77,
                                     10) == dg.DG_ERR_TOO_MANY_LABELS
    assert dg.dg_validate_slots_wide(d, rows, lab, n, 2, 257, 10) == dg.DG_ERR_TOO_MANY_LABELS
    dup = lab.copy()
    dup[0, 76] = 0
    assert dg.dg_validate_slots_wide(d, rows, dup, n, 2, 77, 10) == dg.DG_ERR_LABEL
    # the binding picks the 26-wide or the wide check from the table's width
    dg.validate_slot_table(d, rows, lab, n, 10)
    with pytest.raises(dg.DgError) as ei:
        dg.validate_slot_table(d, rows, dup, n, 10)
    assert ei.value.code == dg.DG_ERR_LABEL


def test_step_set_slots_refuses_bad_tables(lib):
    """The step's slot tables pass the library's synchronous check before they are
    copied: 27 alternatives, a repeated label, an id outside the vocabulary and a
    slot row outside the canvas are refused, and the device tables stay as they were."""
    import torch

    from structured_slot_reads_gb300 import configs, inputs
    from structured_slot_reads_gb300.step import DenoiseStep
    shp = configs.TINY
    w = torch.zeros((shp.V, shp.D), dtype=torch.bfloat16)
    st = DenoiseStep(shp, w, w, device="cpu")
    row, req, lab, n = inputs.slot_table(shp, 0)
    st.set_slots(row, req, lab, n)
    assert st.n_labels.tolist() == n.tolist()
    before = st.label_ids.clone()
    bad_cases = []
    n27 = n.copy()
    n27[0] = 27
    bad_cases.append(((row, req, lab, n27), dg.DG_ERR_TOO_MANY_LABELS))
    dup = lab.copy()
    dup[0, 1] = dup[0, 0]
    bad_cases.append(((row, req, dup, n), dg.DG_ERR_LABEL))
    oov = lab.copy()
    oov[0, 2] = shp.V
    bad_cases.append(((row, req, oov, n), dg.DG_ERR_LABEL))
    bad_cases.append(((np.array([shp.B * shp.C], np.int32), req, lab, n), dg.DG_ERR_SHAPE))
    for args, code in bad_cases:
        with pytest.raises(dg.DgError) as ei:
            st.set_slots(*args)
        assert ei.value.code == code
    assert torch.equal(st.label_ids, before)


def test_two_stage_runner_refuses_27_alternatives(lib):
    """A stage-2 question with 27 items is refused when the batch is set up."""
    import torch

    from structured_slot_reads_gb300 import configs, inputs
    from structured_slot_reads_gb300.read import TwoStageRead
    shp = configs.scaled(configs.MIXED_BATCH, B=2, C=64, P=200, D=256, V=4096)
    tables = inputs.two_stage_tables(shp, 3)
    tables[1]["item_labels"][4] = np.arange(27, dtype=np.int32)
    plen = inputs.prompt_lengths(shp, 3, lo=100)
    w = torch.zeros((shp.V, shp.D), dtype=torch.bfloat16)
    with pytest.raises(dg.DgError) as ei:
        TwoStageRead(shp, w, w, tables, plen, device="cpu", seed=3)
    assert ei.value.code == dg.DG_ERR_TOO_MANY_LABELS


@pytest.mark.parametrize("page_size", [4, 24, 256])
def test_attention_refuses_page_sizes_the_512_kernel_cannot_take(lib, page_size):
    """512-wide heads run only on the tensor-core kernel: a page size it cannot take
    is refused before launch instead of running on another kernel."""
    d = dg.make_dims(B=1, C=64, P_max=96, Hq=8, Hkv=2, d_head=512, W=16)
    ws = dg.dg_workspace_bytes(d, dg.DG_WS_ATTN, 0)
    pages = (96 + page_size - 1) // page_size
    rc = dg.lib().dg_attn_decode(ctypes.byref(d), 256, 256, 256, 256, 256, 256, pages, pages,
                                 page_size, 256, 256, 256, 256, ws, None)
    assert rc == dg.DG_ERR_SHAPE
