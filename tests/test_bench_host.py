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
        assert k == kind in ("step", "read", "two_stage", "prefill", "lmhead", "lmhead_fp8",
                             "mixed", "selfcond", "selfcond_fp8")
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
