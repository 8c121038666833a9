"""The CUDA-core GEMV's unpack identity, checked exactly on the CPU.

The kernel never converts a code to a float.  For a packed word w it ORs
nibble pairs into the mantissa of fp16 1024, which gives 1024 + u for the
even elements (nibbles 0, 2, 4, 6 read as the low nibble of a 16-bit half)
and 1024 + 16 u for the odd ones (read four bits higher), multiplies them by
the activations with exact products, and removes the offsets per 32-weight
chunk with c = 1032 sum_even x + 72 sum_odd x, where q = u - 8:

    sum_i x_i q_i = A + B / 16 - c,
    A = sum_even x_i (1024 + u_i),  B = sum_odd x_i (1024 + 16 u_i).

This file restates that algebra with integer-exact numpy arithmetic (no
kernel code) over every code and random activations, so a sign, offset or
nibble-order slip in the derivation fails here without a GPU."""
import numpy as np


def _fp16_bits_value(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def test_magic_halves_are_exact_offsets():
    for u in range(16):
        lo = _fp16_bits_value(0x6400 | u)              # 1024 + u
        hi = _fp16_bits_value(0x6400 | (u << 4))       # 1024 + 16 u
        assert lo == 1024 + u and hi == 1024 + 16 * u


def test_chunk_identity_over_random_words():
    r = np.random.default_rng(3)
    for _ in range(200):
        words = r.integers(0, 2**32, size=4, dtype=np.uint64)       # one 32-weight chunk
        u = np.array([(int(w) >> (4 * i)) & 0xF for w in words for i in range(8)], np.int64)
        q = u - 8
        x = r.standard_normal(32).astype(np.float16).astype(np.float64)
        direct = float(np.dot(x, q))
        even, odd = np.arange(0, 32, 2), np.arange(1, 32, 2)
        A = float(np.dot(x[even], 1024 + u[even]))
        B = float(np.dot(x[odd], 1024 + 16 * u[odd]))
        c = 1032 * x[even].sum() + 72 * x[odd].sum()
        assert abs((A + B / 16 - c) - direct) <= 1e-9 * (1 + abs(A) + abs(B))


def test_pair_layout_matches_nibble_masks():
    """The masks 0x000F000F and 0x00F000F0 over w and w >> 8 pick, in the two
    halves of each 32-bit register, the nibbles of elements (0, 4), (1, 5),
    (2, 6), (3, 7): the activations are staged in that pair order."""
    r = np.random.default_rng(4)
    for w in r.integers(0, 2**32, size=1000, dtype=np.uint64):
        w = int(w)
        nib = [(w >> (4 * i)) & 0xF for i in range(8)]
        pairs = []
        for src, mask, shift in ((w, 0x000F000F, 0), (w, 0x00F000F0, 4), (w >> 8, 0x000F000F, 0),
                                 (w >> 8, 0x00F000F0, 4)):
            v = src & mask
            pairs.append(((v & 0xFFFF) >> shift, (v >> 16) >> shift))
        assert pairs == [(nib[0], nib[4]), (nib[1], nib[5]), (nib[2], nib[6]), (nib[3], nib[7])]
