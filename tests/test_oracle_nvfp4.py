"""Pins for the oracle's NVFP4 weight quantisation (the 4-bit lm-head operands)."""
import numpy as np

from oracle import nvfp4
from oracle.quant import decode_e4m3
from structured_slot_reads_gb300 import inputs

# the e2m1 magnitudes as the format lists them (codes 0..7; codes 8..15 are their negatives)
PUBLISHED = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_matches_the_published_values():
    vals = [nvfp4.e2m1_value(c) for c in range(16)]
    assert vals[:8] == PUBLISHED
    assert vals[8:] == [-v for v in PUBLISHED]
    assert np.array_equal(nvfp4.decode_e2m1(np.arange(16, dtype=np.uint8)), np.array(vals))


def _brute(y):
    """Nearest of the 16 code values; ties go to the code whose mantissa bit is 0."""
    vals = np.array([nvfp4.e2m1_value(c) for c in range(16)])
    y = min(max(float(y), -6.0), 6.0)
    d = np.abs(vals - y)
    best = [c for c in range(16) if d[c] == d.min()]
    if len(best) > 1:
        best = [c for c in best if (c & 1) == 0] or best
        best = [c for c in best if ((c & 8) != 0) == (y < 0) or nvfp4.e2m1_value(c) == 0] or best
    return nvfp4.e2m1_value(best[0])


def test_rounding_is_nearest_with_ties_to_even_by_brute_force():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rng = np.random.default_rng(0)
    y = np.concatenate([mids, [-m for m in mids], rng.uniform(-7, 7, 3000),
                        [6.0, 6.5, 100.0, -100.0, 0.0, 1e-9]]).astype(np.float32)
    codes = nvfp4.to_e2m1_codes(y)
    for yi, c in zip(y, codes):
        assert nvfp4.e2m1_value(int(c)) == _brute(yi), (yi, c)
    # the ties land on the even mantissa: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2,
    # 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert list(nvfp4.decode_e2m1(codes[:7])) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_quantisation_properties():
    x = inputs.normal_bf16((6, 128), 0.05, 9, 1)
    x[2, 16:32] = 0.0                         # an all-zero block
    x[4] *= 1e-3
    codes, scales, g = nvfp4.quantize_nvfp4(x)
    assert codes.shape == (6, 128) and scales.shape == (6, 8) and codes.max() < 16
    amax = np.abs(x).max()
    assert g == np.float32(amax / np.float32(6 * 448))
    # the tensor's largest element takes the largest block scale and code +-6
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(nvfp4.e2m1_value(codes[r, c])) == 6.0
    assert decode_e4m3(scales[r, c // 16:c // 16 + 1])[0] == 448.0
    assert np.all(codes[2, 16:32] == 0) and scales[2, 1] == 0
    deq = nvfp4.dequantize_nvfp4(codes, scales, g)
    s = np.repeat(decode_e4m3(scales), 16, axis=1) * float(g)
    y = np.where(s > 0, x / np.where(s > 0, s, 1), 0)
    # within half an e2m1 step of the element's magnitude (steps 0.5, 1, 2), in units of s g
    step = np.where(np.abs(y) < 2, 0.5, np.where(np.abs(y) < 4, 1.0, 2.0))
    assert np.all(np.abs(deq - x) <= step / 2 * s * (1 + 1e-6) + 1e-30)
    # sign symmetry
    cn, sn, gn = nvfp4.quantize_nvfp4(-x)
    assert gn == g and np.array_equal(sn, scales)
    assert np.array_equal(nvfp4.dequantize_nvfp4(cn, sn, gn), -deq)
    # packing round trips (plain and the K-block-major layout of the CUDA quantiser)
    assert np.array_equal(nvfp4.unpack_nibbles(nvfp4.pack_nibbles(codes)), codes)
    ckb, skb = nvfp4.to_kblock_layout(codes, scales)
    assert ckb.shape == (2, 6, 32) and skb.shape == (2, 6, 4)
    assert ckb[1, 3, 5] == (codes[3, 64 + 10] | (codes[3, 64 + 11] << 4))
    assert skb[1, 4, 2] == scales[4, 4 + 2]
    back_c, back_s = nvfp4.from_kblock_layout(ckb, skb)
    assert np.array_equal(back_c, codes) and np.array_equal(back_s, scales)
    # a slice quantised with the whole tensor's scale gives the same rows
    c2, s2, g2 = nvfp4.quantize_nvfp4(x[2:5], g=g)
    assert g2 == g and np.array_equal(c2, codes[2:5]) and np.array_equal(s2, scales[2:5])


def test_zero_tensor():
    codes, scales, g = nvfp4.quantize_nvfp4(np.zeros((2, 32), np.float32))
    assert g == 1.0 and not codes.any() and not scales.any()


def test_values_on_the_grid_quantise_exactly():
    """A tensor whose blocks are e2m1 values times a block scale that is an e4m3 value
    times a power-of-two tensor scale g = 2^-6 (the largest block reaching
    6 * 448 * g, so g comes out exactly): every element comes back exactly."""
    rng = np.random.default_rng(3)
    vals = np.array(PUBLISHED + [-v for v in PUBLISHED[1:]])
    blocks = rng.choice(vals, size=(4, 64))
    blocks[:, ::16] = 6.0                    # each block reaches 6
    bs = 2.0 ** rng.integers(-3, 3, size=(4, 4))
    bs[0, 0] = 448.0 * 2.0 ** -6             # the tensor's largest block
    x = (blocks * np.repeat(bs, 16, axis=1)).astype(np.float32)
    codes, scales, g = nvfp4.quantize_nvfp4(x)
    assert g == 2.0 ** -6
    assert np.array_equal(nvfp4.decode_e2m1(codes), blocks)
    assert np.array_equal(nvfp4.dequantize_nvfp4(codes, scales, g), x.astype(np.float64))


def test_mma_layout_places_each_scale_by_its_definition():
    """The block-scaled layout.  Scale atoms: row 32 j + l of a 128-row tile, 64-value
    step k, block q of the step at atom [tile][k], byte 16 l + 4 j + q; rows past R
    scale 0.  Codes two a byte, the even element low, in 128 x 128-byte blocks per
    (128-row tile, 256-value K block): element k of row r in byte (k % 256) // 2 of
    row r % 128 of block (r // 128, k // 256), zero past R and past K.  Checked
    byte by byte against that definition (a ragged last K block: K = 320), then
    the inverse."""
    R, K = 130, 320
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, (R, K), dtype=np.uint8)
    scales = rng.integers(0, 256, (R, K // 16), dtype=np.uint8)
    packed, atoms = nvfp4.to_mma_layout(codes, scales)
    assert packed.shape == (2, 2, 128, 128) and atoms.shape == (2, 5, 512)
    for r in range(R):
        for k in range(0, K, 2):
            byte = packed[r // 128, k // 256, r % 128, (k % 256) // 2]
            assert byte == codes[r, k] | (codes[r, k + 1] << 4)
    assert packed[1, :, 2:, :].sum() == 0              # rows 130..255
    assert packed[:, 1, :, 32:].sum() == 0             # values 320..511 of block 1
    for r in range(R):
        t, rr = divmod(r, 128)
        j, l = divmod(rr, 32)
        for b in range(K // 16):
            k, q = divmod(b, 4)
            assert atoms[t, k, 16 * l + 4 * j + q] == scales[r, b]
    assert atoms[1, :, 16 * 2:].sum() == 0            # rows 130..255 of tile 1
    assert atoms[1, :, 4:16].sum() == 0               # rows 160, 192, 224 (j > 0, l = 0)
    c2, s2 = nvfp4.from_mma_layout(packed, atoms, R)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
