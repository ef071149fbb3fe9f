"""Philox4x32-10 counter-based generator, written from its published definition.

TEST INFRASTRUCTURE ONLY: this module belongs to the CPU oracle.  Only the test
suite, the smoke check and the CPU-baseline leg of the benchmark may import it;
the product (the CUDA library and its binding) never does.

Definition followed: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 3.2 (the Philox
bijection) with the N=4, W=32 constants of its Table 2.  One round maps the
counter (x0, x1, x2, x3) under round key (k0, k1) to

    (hi(M1*x2) ^ x1 ^ k0,  lo(M1*x2),  hi(M0*x0) ^ x3 ^ k1,  lo(M0*x0))

where hi/lo are the upper and lower 32 bits of the 64-bit product; the round
key advances by the Weyl increments (W0, W1) between rounds; ten rounds.

How the structured-read method uses it (the DiffusionGemma pages only say the
canvas starts from noise / random placeholder tokens and that the server
re-reads a slot with fresh noise draws; they do not fix a generator): the
64-bit seed is the key (low word k0, high word k1) and the counter is
(request, step, draw, slot).  The first output word, shifted right so that
its top log2(V) bits remain, is the noise token id (V a power of two, so the
map is exactly uniform).
"""
import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """Apply Philox4x32 with 10 rounds.

    ctr: uint32 array of shape [..., 4]; key: uint32 array broadcastable to [..., 2].
    Returns uint32 [..., 4].
    """
    ctr = np.asarray(ctr, dtype=np.uint32)
    key = np.asarray(key, dtype=np.uint32)
    x0, x1, x2, x3 = (ctr[..., i].astype(np.uint64) for i in range(4))
    k0 = key[..., 0].astype(np.uint64)
    k1 = key[..., 1].astype(np.uint64)
    m0 = np.uint64(M0)
    m1 = np.uint64(M1)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(W0)) & _MASK
            k1 = (k1 + np.uint64(W1)) & _MASK
        p0 = m0 * x0          # < 2^64: product of two 32-bit values
        p1 = m1 * x2
        y0 = (p1 >> np.uint64(32)) ^ x1 ^ k0
        y1 = p1 & _MASK
        y2 = (p0 >> np.uint64(32)) ^ x3 ^ k1
        y3 = p0 & _MASK
        x0, x1, x2, x3 = y0, y1, y2, y3
    return np.stack([x0, x1, x2, x3], axis=-1).astype(np.uint32)


def seed_key(seed):
    """Split a 64-bit seed into the Philox key (k0 = low word, k1 = high word)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)


def noise_tokens(seed, req, step, n_draws, n_slots, vocab):
    """Noise token ids [n_draws, n_slots] for one request and one denoise step.

    Counter = (req, step, draw r, slot s); token = word0 >> (32 - log2 V).
    """
    vocab = int(vocab)
    if vocab <= 1 or vocab & (vocab - 1):
        raise ValueError("vocab must be a power of two > 1 for the noise map")
    bits = vocab.bit_length() - 1
    r = np.arange(n_draws, dtype=np.uint32)[:, None]
    s = np.arange(n_slots, dtype=np.uint32)[None, :]
    ctr = np.stack(np.broadcast_arrays(np.uint32(req), np.uint32(step), r, s), axis=-1)
    out = philox4x32_10(ctr, seed_key(seed))
    return (out[..., 0] >> np.uint32(32 - bits)).astype(np.int64)
