"""e4m3 operands of the 8-bit lm-head pass (test infrastructure, like the rest of oracle/).

tau-home.com, "DiffusionGemma like Jev" ("Running NVFP4 locally with a
Jev-compatible System One endpoint") and 24-ai.news, "DiffusionGemma integrated
into vLLM" ("Measured performance": an FP8 checkpoint with dynamic activation
scaling): the model runs on 8-bit weights and activations.

Reading: one fp32 scale per row, scale = amax|x| / 448 (the largest finite
e4m3 value; 1 for an all-zero row), q = e4m3(x / scale) with fp32 division and
round-to-nearest-even; the 8-bit lm-head pass computes the plain lm-head
statistics (``lmhead_stats``) of the dequantised operands q * scale.
The e4m3 cast is torch's (a library routine); the tests pin it against the
format's definition by brute force.
"""
import numpy as np
import torch

E4M3_MAX = 448.0


def e4m3_value(byte):
    """Value of one e4m3 (fn) bit pattern by the format's definition: sign, 4-bit
    exponent with bias 7, 3-bit mantissa, subnormals at exponent 0, no infinities,
    S.1111.111 is NaN."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def to_e4m3_bytes(y):
    """float32 array -> e4m3 bit patterns (uint8), round to nearest even (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def decode_e4m3(q):
    """uint8 e4m3 bit patterns -> float64 values (torch's decode)."""
    t = torch.from_numpy(np.ascontiguousarray(q, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def quantize_rows_e4m3(x):
    """Per-row e4m3 quantisation of a bf16-valued float32 matrix [R, C].

    Returns (q uint8 [R, C], scale float32 [R])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / scale[:, None]).astype(np.float32)
    return to_e4m3_bytes(y), scale


def dequantize_rows(q, scale):
    """q * scale per row, float64."""
    return decode_e4m3(q) * np.asarray(scale, np.float64)[:, None]


def quantize_cols_e4m3(x):
    """Per-column e4m3 quantisation of a bf16-valued float32 matrix [R, C], stored
    transposed: column c of x is row c of the result.

    Returns (qt uint8 [C, R], scale float32 [C]) with scale[c] = amax_r |x[r, c]| / 448
    (1 for a zero column) and qt[c, r] = e4m3(x[r, c] / scale[c])."""
    return quantize_rows_e4m3(np.ascontiguousarray(np.asarray(x, np.float32).T))


def selfcond_fp8(p8, p_scale, row_scale, e8t, e_scale):
    """Expected embedding on 8-bit operands, float64.

    24-ai.news, "Token commit mechanism": e_i = sum_v p_iv E[v].  With the
    probabilities quantised per row (p8, p_scale; row_scale the row's 1/S, or
    None for 1) and E quantised per d_model column and transposed (e8t, e_scale):
    out[i, c] = row_scale[i] * p_scale[i] * e_scale[c] * sum_v p8[i, v] e8t[c, v]."""
    p = decode_e4m3(p8)
    et = decode_e4m3(e8t)
    rs = np.asarray(p_scale, np.float64)
    if row_scale is not None:
        rs = rs * np.asarray(row_scale, np.float64)
    return rs[:, None] * (p @ et.T) * np.asarray(e_scale, np.float64)[None, :]
