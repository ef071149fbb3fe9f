"""Pins for the oracle's e4m3 quantisation (8-bit lm-head operands)."""
import numpy as np

import oracle
from oracle import quant
from structured_slot_reads_gb300 import inputs


def _all_values():
    return np.array([quant.e4m3_value(b) for b in range(256)])


def test_decode_matches_the_format_definition():
    """torch's e4m3 decode equals the sign/exponent/mantissa definition on all 256 patterns."""
    ref = _all_values()
    got = quant.decode_e4m3(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(ref) == 448.0 and np.nanmin(ref) == -448.0


def test_cast_is_nearest_with_ties_to_even_by_brute_force():
    vals = _all_values()
    finite = np.where(~np.isnan(vals))[0]
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1e-2, 2000),
                        (vals[finite][:-1] + vals[finite][1:]) / 2]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    got = quant.to_e4m3_bytes(x)
    for xi, g in zip(x, got):
        d = np.abs(vals[finite] - float(xi))
        best = finite[d == d.min()]
        if len(best) > 1:  # a tie: the even mantissa (lowest bit 0), same sign as x
            best = [b for b in best if (b & 1) == 0 and ((b & 0x80) != 0) == (xi < 0)] or best
        assert quant.e4m3_value(int(g)) == quant.e4m3_value(int(best[0])), (xi, g, best)


def test_quantize_rows_properties():
    x = inputs.normal_bf16((8, 300), 1.0, 5, 1)
    x[3] = 0.0
    x[5] *= 1e-3
    q, scale = oracle.quantize_rows_e4m3(x)
    deq = oracle.dequantize_rows(q, scale)
    assert scale[3] == 1.0 and np.all(deq[3] == 0)
    for r in range(8):
        if r == 3:
            continue
        a = np.argmax(np.abs(x[r]))
        assert abs(quant.decode_e4m3(q[r, a:a + 1])[0]) == 448.0   # the row's amax maps to 448
        big = np.abs(x[r]) > scale[r] * 2.0 ** -6          # normal e4m3 range
        err = np.abs(deq[r] - x[r])
        assert np.all(err[big] <= 2.0 ** -4 * np.abs(x[r][big]) * (1 + 1e-7))
    qn, sn = oracle.quantize_rows_e4m3(-x)
    assert np.array_equal(sn, scale) and np.array_equal(oracle.dequantize_rows(qn, sn), -deq)


def test_fp8_lmhead_reduces_to_the_plain_statistics_of_the_dequantised_operands():
    """With operands already on the e4m3 grid (scale 1), quantisation is exact."""
    rng = np.random.default_rng(1)
    vals = _all_values()
    grid = vals[np.isfinite(vals) & (np.abs(vals) <= 2)]
    h = rng.choice(grid, (4, 64)).astype(np.float32)
    h[:, 0] = 448.0  # amax 448: scale exactly 1
    q, scale = oracle.quantize_rows_e4m3(h)
    assert np.all(scale == 1.0) and np.array_equal(oracle.dequantize_rows(q, scale), h)
