"""NVFP4 weights of the 4-bit lm-head pass (test infrastructure, like the rest of oracle/).

tau-home.com, "DiffusionGemma like Jev" ("Running NVFP4 locally with a
Jev-compatible System One endpoint") and agentlenshq.com, "4x faster via
parallel diffusion" ("Architecture": NVFP4 kernels for Hopper and Blackwell)
run the model on NVFP4 weights.  The pages name the format, not its layout;
the reading taken here is the format as NVIDIA's Blackwell documentation
defines it:

* elements: e2m1 (1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit;
  magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte, the even element of a
  pair in the low nibble;
* one e4m3 scale per 16 consecutive elements of a row;
* one fp32 scale per tensor.

Quantisation recipe (fp32 arithmetic throughout, so that the CUDA quantiser and
this one take the same decisions): tensor scale g = amax|x| / (6 * 448) (1 for
an all-zero tensor); for each block of 16, s = e4m3((amax_block / 6) / g)
(round to nearest even, saturating at 448); element codes
e2m1(x / (s_value * g)) (round to nearest, ties to the even mantissa,
saturating at 6), all codes 0 for a block whose scale is 0.  The dequantised
weight is e2m1 * s * g; the lm-head pass multiplies the rows by e2m1 * s
(exact in bf16) and applies g with the temperature.
"""
import numpy as np

from .quant import decode_e4m3, to_e4m3_bytes

E2M1_MAX = 6.0
BLOCK = 16


def e2m1_value(code):
    """Value of a 4-bit e2m1 code by the format's definition."""
    code = int(code) & 0xF
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * 0.5 * m
    return s * (1.0 + 0.5 * m) * 2.0 ** (e - 1)


_MAGS = np.array([e2m1_value(c) for c in range(8)])   # codes 0..7: 0, .5, 1, 1.5, 2, 3, 4, 6


def to_e2m1_codes(y):
    """float32 array -> e2m1 codes (uint8 0..15): nearest magnitude, ties to the code
    with an even mantissa bit, saturating at 6; the sign bit follows y (0 for +0)."""
    y = np.asarray(y, dtype=np.float32)
    a = np.minimum(np.abs(y).astype(np.float64), E2M1_MAX)
    d = np.abs(a[..., None] - _MAGS)                      # [..., 8]
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # among tied codes prefer an even mantissa bit (code & 1 == 0)
    even = cand & ((np.arange(8) & 1) == 0)
    pick = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    sign = (np.signbit(y) & (pick > 0)).astype(np.uint8) << 3
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


def decode_e2m1(codes):
    """e2m1 codes -> float64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = _MAGS[codes & 0x7]
    return np.where(codes & 0x8, -mag, mag)


def tensor_scale(amax):
    """g = amax / (6 * 448) in fp32, 1 for an all-zero tensor."""
    amax = np.float32(amax)
    return np.float32(amax / np.float32(E2M1_MAX * 448.0)) if amax > 0 else np.float32(1.0)


def quantize_nvfp4(x, g=None):
    """NVFP4 quantisation of a bf16-valued float32 matrix [R, K] (K a multiple of 16).

    ``g`` (optional) is the tensor scale when x is a slice of a larger tensor.
    Returns (codes uint8 [R, K] one code per element, scales uint8 [R, K / 16] e4m3
    bit patterns, g float32 tensor scale)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    assert K % BLOCK == 0
    if g is None:
        g = tensor_scale(np.abs(x).max() if x.size else 0.0)
    g = np.float32(g)
    xb = x.reshape(R, K // BLOCK, BLOCK)
    bmax = np.abs(xb).max(axis=2)
    s_code = to_e4m3_bytes(((bmax / np.float32(E2M1_MAX)).astype(np.float32) / g)
                           .astype(np.float32))
    s_val = decode_e4m3(s_code).astype(np.float32)
    denom = (s_val * g).astype(np.float32)
    safe = np.where(denom > 0, denom, np.float32(1.0)).astype(np.float32)
    y = (xb / safe[..., None]).astype(np.float32)
    codes = to_e2m1_codes(y)
    codes = np.where((denom > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(R, K), s_code.astype(np.uint8), g


def pack_nibbles(codes):
    """[R, K] codes -> [R, K / 2] bytes, element 2i in the low nibble of byte i."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def block_values(codes, scales):
    """e2m1 * block scale, float64 [R, K]: what the pass multiplies the rows by."""
    v = decode_e2m1(codes)
    s = decode_e4m3(scales)
    return v * np.repeat(s, BLOCK, axis=1)


def dequantize_nvfp4(codes, scales, g):
    """The dequantised weight e2m1 * s * g, float64 [R, K]."""
    return block_values(codes, scales) * float(g)


def to_kblock_layout(codes, scales):
    """The K-block-major layout of the CUDA quantiser: codes [K/64][R][32] bytes (two
    codes a byte, the even element low) and scales [K/64][R][4]."""
    R, K = codes.shape
    nkb = K // 64
    packed = pack_nibbles(codes).reshape(R, nkb, 32).transpose(1, 0, 2)
    sc = np.asarray(scales, np.uint8).reshape(R, nkb, 4).transpose(1, 0, 2)
    return np.ascontiguousarray(packed), np.ascontiguousarray(sc)


def from_kblock_layout(codes_kb, scales_kb):
    """Inverse of to_kblock_layout: codes [R, K], scales [R, K / 16]."""
    nkb, R, _ = codes_kb.shape
    packed = np.ascontiguousarray(np.asarray(codes_kb, np.uint8).transpose(1, 0, 2)).reshape(R, -1)
    sc = np.ascontiguousarray(np.asarray(scales_kb, np.uint8).transpose(1, 0, 2)).reshape(R, -1)
    return unpack_nibbles(packed), sc


def to_mma_layout(codes, scales):
    """The layout of the block-scaled pass (dg_quantize_nvfp4_mma).  Codes two a
    byte (the even element low) in 128 x 128-byte blocks, one per (128-row tile,
    256-value K block): [ceil(R/128)][ceil(K/256)][128][128], element k of row v in
    byte (k % 256) / 2 of row v % 128 of block (v // 128, k // 256), zero past R
    rows and past K.  Scales as 512-byte atoms [ceil(R/128)][K/64][512]: row
    32 j + l of a 128-row tile has the four scales of a 64-value step (its blocks of
    16 in order) at bytes 16 l + 4 j .. 16 l + 4 j + 3; rows past R have scale 0."""
    R, K = codes.shape
    nks = K // 64
    nkb = (nks + 3) // 4
    tiles = (R + 127) // 128
    sc = np.zeros((tiles * 128, nks, 4), np.uint8)
    sc[:R] = np.asarray(scales, np.uint8).reshape(R, nks, 4)
    sc = sc.reshape(tiles, 4, 32, nks, 4)                 # [tile][j][l][step][block]
    atoms = sc.transpose(0, 3, 2, 1, 4)                   # [tile][step][l][j][block]
    flat = np.zeros((tiles * 128, nkb * 128), np.uint8)
    flat[:R, :K // 2] = pack_nibbles(codes)
    blocks = flat.reshape(tiles, 128, nkb, 128).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(blocks), np.ascontiguousarray(atoms).reshape(tiles, nks, 512)


def from_mma_layout(packed, atoms, R):
    """Inverse of to_mma_layout: codes [R, K], scales [R, K / 16]."""
    tiles, nks, _ = atoms.shape
    nkb = (nks + 3) // 4
    a = np.asarray(atoms, np.uint8).reshape(tiles, nks, 32, 4, 4)
    sc = a.transpose(0, 3, 2, 1, 4).reshape(tiles * 128, nks * 4)
    blocks = np.asarray(packed, np.uint8).reshape(tiles, nkb, 128, 128)
    flat = blocks.transpose(0, 2, 1, 3).reshape(tiles * 128, nkb * 128)
    return unpack_nibbles(flat[:R, :nks * 32]), np.ascontiguousarray(sc[:R])
