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


def test_quantize_cols_properties():
    """Column c of x becomes row c of qt with its own scale: the column's largest
    magnitude maps to +-448, a zero column keeps scale 1, and the dequantised
    values lie within half an e4m3 step of x (relative 2^-4 in the normal range)."""
    x = inputs.normal_bf16((300, 8), 1.0, 5, 2)
    x[:, 2] = 0.0
    x[:, 6] *= 1e-3
    qt, scale = oracle.quantize_cols_e4m3(x)
    assert qt.shape == (8, 300) and scale.shape == (8,)
    assert scale[2] == 1.0 and np.all(quant.decode_e4m3(qt[2]) == 0)
    for c in range(8):
        if c == 2:
            continue
        assert scale[c] == np.float32(np.abs(x[:, c]).max()) / np.float32(448.0)
        a = np.argmax(np.abs(x[:, c]))
        assert quant.decode_e4m3(qt[c, a:a + 1])[0] == 448.0 * np.sign(x[a, c])
        deq = quant.decode_e4m3(qt[c]) * float(scale[c])
        big = np.abs(x[:, c]) > scale[c] * 2.0 ** -6
        err = np.abs(deq - x[:, c])
        assert np.all(err[big] <= 2.0 ** -4 * np.abs(x[big, c]) * (1 + 1e-7))
    # bytes built column by column with the format's own cast
    for c in (0, 5):
        y = (x[:, c] / scale[c]).astype(np.float32)
        assert np.array_equal(qt[c], quant.to_e4m3_bytes(y))


def _fp8_operands(V=64, D=12, seed=3):
    e = inputs.normal_bf16((V, D), 0.2, seed, 3)
    e8t, e_scale = oracle.quantize_cols_e4m3(e)
    e_deq = (quant.decode_e4m3(e8t) * e_scale[:, None].astype(np.float64)).T   # [V, D]
    return e8t, e_scale, e_deq


def test_selfcond_fp8_one_hot_row_is_the_dequantised_embedding_row():
    """A probability row with all mass on v* (byte 448, p_scale 1/448) returns
    row_scale * E_deq[v*] exactly."""
    V, D = 64, 12
    e8t, e_scale, e_deq = _fp8_operands(V, D)
    p8 = np.zeros((3, V), np.uint8)
    vstar = [0, 17, 63]
    for i, v in enumerate(vstar):
        p8[i, v] = 0x7E                     # +448
    p_scale = np.full(3, 1.0 / 448.0, np.float32)
    rs = np.array([1.0, 0.5, 2.0], np.float32)
    out = oracle.selfcond_fp8(p8, p_scale, rs, e8t, e_scale)
    for i, v in enumerate(vstar):
        np.testing.assert_allclose(out[i], float(rs[i]) * float(p_scale[i]) * 448.0 * e_deq[v],
                                   rtol=1e-12, atol=1e-15)


def test_selfcond_fp8_uniform_row_is_the_column_mean():
    """Equal probabilities (every byte 448, p_scale 1/(448 V)) give the column mean
    of E_deq; a zero row gives zero."""
    V, D = 64, 12
    e8t, e_scale, e_deq = _fp8_operands(V, D, seed=4)
    p8 = np.full((2, V), 0x7E, np.uint8)
    p8[1] = 0
    p_scale = np.full(2, 1.0 / (448.0 * V), np.float64)
    out = oracle.selfcond_fp8(p8, p_scale, None, e8t, e_scale)
    np.testing.assert_allclose(out[0], e_deq.mean(axis=0), rtol=1e-12, atol=1e-15)
    assert np.all(out[1] == 0)
