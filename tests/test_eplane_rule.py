"""CPU check of the E1M2 two-plane split that the GEMM relies on.

Read as an E2M1 code, an E1M2 nibble m has the value R(m) in
{0, .5, 1, 1.5, 2, 3, 4, 6}; the correction plane holds E(m) in
{0, .5, 1, 1.5, 2, 2, 2, 1} as E2M1 codes with the same sign, so that
R(m) + E(m) = m and the E1M2 value m/2 is (R + E)/2 (include/ufp4.h, the
eplane field).  The plane of a packed word is documented as a bit mask: per
nibble s|b2 b1 b0, bit 0 is kept iff !b2, bit 1 iff (!b2 | b0), bit 2 iff
!(b0 & b1), the sign always.  This test restates that mask on whole 32-bit
words (eight nibbles at once, as the quantizer and the GEMM apply it) and
checks it against the per-nibble decomposition for all 16 codes and for
random words.
"""
import numpy as np

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
M = 0xFFFFFFFF


def plane_word(w):
    """The documented mask, applied to eight packed nibbles at once."""
    u, v, t, x = w >> 1, (w << 1) & M, w >> 2, (w << 2) & M
    keep = ((~t & 0x11111111) | ((~u | v) & 0x22222222) | (~(x & v) & 0x44444444) | 0x88888888) & M
    return w & keep


def test_split_of_every_code():
    for code in range(16):
        e = plane_word(code) & 0xF
        m, em = code & 7, e & 7
        assert (e & 8) == (code & 8)                      # sign kept
        assert E2M1[m] + E2M1[em] == m, (code, e)         # R + E = 2 * (m / 2)
    # the E plane takes the documented values
    assert [E2M1[plane_word(m) & 7] for m in range(8)] == [0, .5, 1, 1.5, 2, 2, 2, 1]


def test_packed_words_match_per_nibble_rule():
    rng = np.random.default_rng(3)
    words = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64)
    for w in words.tolist():
        p = plane_word(w)
        for j in range(8):
            c, e = (w >> (4 * j)) & 0xF, (p >> (4 * j)) & 0xF
            if E2M1[c & 7] + E2M1[e & 7] != (c & 7) or (c & 8) != (e & 8):
                raise AssertionError((hex(w), j))
