"""The packed code layouts of include/lq.h, packed here from the header's text and
read back by the unpacker the GPU parity tests use (no GPU involved)."""
import numpy as np

from tests._gpu import unpack_codes


def _pack6(c):
    """c int [rows][128] in [-31, 31] -> uint8 [rows][96] per the 6-bit layout."""
    v = (c + 32).astype(np.uint32)
    rows = c.shape[0]
    out = np.zeros((rows, 96), np.uint8)
    for i in range(rows):
        for j in range(128):
            lo = v[i, j] & 15
            out[i, j // 2] |= lo << (4 * (j % 2))  # code 2j' in the low nibble
            blk, e = divmod(j, 16)
            g, b = 2 * (e // 8) + e % 2, (e % 8) // 2
            bit = 8 * b + 2 * g
            word = int.from_bytes(out[i, 64 + 4 * blk:68 + 4 * blk].tobytes(), "little")
            word |= int(v[i, j] >> 4) << bit
            out[i, 64 + 4 * blk:68 + 4 * blk] = np.frombuffer(word.to_bytes(4, "little"), np.uint8)
    return out


def _pack4(c):
    v = (c + 8).astype(np.uint8)
    return (v[:, 0::2] | (v[:, 1::2] << 4)).astype(np.uint8)


def test_6bit_rows_round_trip():
    rng = np.random.default_rng(3)
    c = rng.integers(-31, 32, size=(7, 128))
    c[0] = np.arange(128) % 63 - 31  # every value, every position class
    assert np.array_equal(unpack_codes(_pack6(c)), c.astype(np.int8))


def test_4bit_rows_round_trip():
    rng = np.random.default_rng(4)
    c = rng.integers(-7, 8, size=(5, 128))
    assert np.array_equal(unpack_codes(_pack4(c)), c.astype(np.int8))
