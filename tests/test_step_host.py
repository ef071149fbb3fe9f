"""Host-side layout of the step's input and decision arenas (no GPU needed)."""
import pytest

torch = pytest.importorskip("torch")

from structured_slot_reads_gb300.step import Buffers, _carve, _layout  # noqa: E402


def test_arena_views_are_aligned_disjoint_and_round_trip():
    specs = [("h0", (3, 5), torch.bfloat16), ("inv_t", (3,), torch.float32),
             ("q", (2, 3, 4, 8), torch.bfloat16), ("cand", (2, 3), torch.uint8),
             ("empty", (0, 4), torch.bfloat16), ("tok", (7,), torch.int32)]
    lay = _layout(specs)
    entries, total = lay
    spans = []
    for name, shape, dt, off, nb in entries:
        assert off % 256 == 0
        spans.append((off, off + nb))
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= total
    a, b = _carve(lay, "cpu"), _carve(lay, "cpu")
    assert isinstance(a, Buffers) and a.arena.numel() == total
    for name, shape, dt, off, nb in entries:
        t = a[name]
        assert t.shape == shape and t.dtype == dt and t.is_contiguous()
        if t.numel():
            t.copy_(torch.arange(t.numel()).reshape(shape).to(dt))
    b.arena.copy_(a.arena)                  # one copy moves the whole set
    for name in a:
        assert torch.equal(a[name], b[name])
