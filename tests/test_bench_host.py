"""Host-side checks of bench.py: the workload table and its work counts."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_workload_resolves_to_a_shape():
    b = _bench()
    for name, (kind, _, kw) in b.WORKLOADS.items():
        k, shape = b.workload_shape(name)
        assert k == kind in ("step", "read", "read_fp4", "two_stage", "prefill", "lmhead",
                             "lmhead_fp8",
                             "lmhead_fp4", "lmhead_fp4mma", "mixed", "selfcond", "selfcond_fp8",
                             "heads", "heads_fp8")
        for f, v in kw.items():
            assert getattr(shape, f) == v
    assert b.workload_shape("sweep_read_b64")[1].B == 64
    assert b.workload_shape("long_context_read")[1].P == 110707


def test_attention_work_counts_visible_keys():
    """attn_flops = 4 Hq d x (number of visible (row, key) pairs), counted by brute force."""
    from structured_slot_reads_gb300 import configs
    b = _bench()
    shape = configs.scaled(configs.TINY, B=3)
    plen = np.array([64, 10, 0])
    C, W = shape.C, shape.W
    pairs = 0
    for p in plen:
        for i in range(C):
            pairs += p + sum(1 for j in range(C) if abs(i - j) <= W)
    assert b.attn_flops(shape, plen) == 4.0 * shape.Hq * shape.d_head * pairs
    assert b.attn_flops(shape) == b.attn_flops(shape, [shape.P] * 3)
    kv = (plen.sum() + 3 * C) * shape.Hkv * shape.d_head * 4
    assert b.attn_bytes(shape, plen) == kv + 2 * 3 * C * shape.Hq * shape.d_head * 2


def test_prefill_work_counts_causal_pairs():
    from structured_slot_reads_gb300 import configs
    b = _bench()
    shape = configs.scaled(configs.TINY, B=2, P=9, Hq=4, d_head=64)
    pairs = sum(1 for i in range(9) for j in range(9) if j <= i)
    assert b.prefill_flops(shape) == 4.0 * 2 * 4 * 64 * pairs


def test_reference_arm_times_whole_oracle_steps():
    """The reference arm times whole float64 steps (no sampling) and reports the
    steps it actually timed; at the tiny shape every part runs in milliseconds."""
    import argparse

    from structured_slot_reads_gb300 import configs
    b = _bench()
    line = b.reference_arm(argparse.Namespace(steps=3, warmup=5), 0, shape=configs.TINY)
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 2
    assert line["steps_requested"] == 3 and line["warmup_requested"] == 5
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert set(line["cpu_baseline"]["parts_s"]) == {"attention", "lmhead", "slot_read", "commit",
                                                   "selfcond", "canvas_update"}
    # a tiny time budget stops after the first timed step
    short = b.reference_arm(argparse.Namespace(steps=50, warmup=0), 0, budget_s=0.0,
                            shape=configs.TINY)
    assert short["steps"] == 1 and short["warmup"] == 0
    assert b.reference_arm(argparse.Namespace(steps=3, warmup=5), 1) is None


def test_heads_roofline_counts_algorithmic_bytes():
    """The heads pass's algorithmic bytes are W plus the rows and statistics; the
    bf16 probability hand-off to the P.E GEMM is reported apart."""
    from structured_slot_reads_gb300 import configs
    b = _bench()
    shape = configs.FULL_CANVAS

    class St:
        n_draw, S = 12, 3
    work = b.call_work(shape, St())
    W = shape.V * shape.D * 2
    by, fl = work["dg_denoise_heads"]
    assert W < by < W * 1.002
    assert fl == 2.0 * (256 + 12) * shape.V * shape.D
    assert b.spill_bytes(shape) == 256 * shape.V * 2
    assert work["dg_selfcond_from_probs"][0] < W * 1.01
    assert work["dg_commit"][0] > 0 and work["dg_slot_finish"][0] > 0
