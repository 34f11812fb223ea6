"""Pins for the oracle's b-bit GEMV (b = 2..8; BaseRT §3.3, §4.1: kernels per
quantisation format).  The packing reading: code k of a row in bits
b*k .. b*k+b-1 of the row's little-endian bit stream, a code crossing a word
boundary continuing in the next word.  Pinned by a hand-packed word, the
generator's own codes (numpy packbits against the oracle's shift-and-mask),
equality with the pinned 4- and 8-bit oracles, one-hot probes of every code
at word-crossing positions, and exact rational brute force; the planted
mistakes (an off-by-one bit offset, dropped high bits of a crossing code)
each fail a pin."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import q4synth

BITS = (2, 3, 4, 5, 6, 8)


def test_hand_packed_3bit_word():
    """Codes 1,2,3,4,5,6,7,0,1,2,7 at 3 bits: word 0 = 0xd11f58d1 (code 10's
    low two bits in bits 30-31), word 1 = 0x1 (its high bit)."""
    row = np.array([0xD11F58D1, 0x1, 0x0], np.uint32)
    assert [oracle.codeb(row, k, 3) for k in range(11)] == [1, 2, 3, 4, 5, 6, 7, 0, 1, 2, 7]
    assert [oracle.codeb(row, k, 3, mutant=10) for k in range(11)][10] == 3     # high bit lost
    assert [oracle.codeb(row, k, 3, mutant=9) for k in range(11)][:3] != [1, 2, 3]


@pytest.mark.parametrize("bits", BITS)
def test_oracle_reads_the_generators_codes(bits):
    m = q4synth.qb_matrix(800 + bits, 3, 256, bits)
    for n in range(3):
        got = [oracle.codeb(m.Wq[n], k, bits) for k in range(256)]
        assert got == m.codes[n].tolist()


def test_four_and_eight_bits_coincide_with_the_pinned_layouts():
    m4 = q4synth.q4_matrix(810, 40, 320)
    x = q4synth.activations(811, 3, 320)
    assert np.array_equal(oracle.gemvb(m4.Wq, m4.scales, m4.biases, x, 4)[0], oracle.gemv(m4.Wq, m4.scales, m4.biases, x)[0])
    m8 = q4synth.q8_matrix(812, 40, 320)
    assert np.array_equal(oracle.gemvb(m8.Wq, m8.scales, m8.biases, x, 8)[0],
                          oracle.gemv8(m8.Wq, m8.scales, m8.biases, x)[0])


@pytest.mark.parametrize("bits", (2, 3, 5, 6))
def test_one_hot_every_code_at_crossing_positions(bits):
    """Row with code c at position j and code 0 elsewhere, x = e_j:
    y = s c + b exactly (s = 2^-4, b = -0.5).  The positions include every
    code that crosses a word boundary in the first 128."""
    K = 128
    cross = [k for k in range(K) if (bits * k) % 32 + bits > 32]
    positions = sorted(set(cross + [0, 1, 31, K - 1]))
    s = np.full((1, K // 64), 2.0 ** -4, np.float16)
    b = np.full((1, K // 64), -0.5, np.float16)
    for j in positions:
        x = np.zeros((1, K), np.float16)
        x[0, j] = 1.0
        for c in range(1 << bits):
            codes = np.zeros((1, K), np.uint32)
            codes[0, j] = c
            Wq = q4synth.pack_codes(codes, bits)
            y, _ = oracle.gemvb(Wq, s, b, x, bits)
            assert y[0, 0] == 2.0 ** -4 * c - 0.5, (bits, j, c)
    # the mistakes fail here (2-bit codes never cross a word boundary)
    codes = np.zeros((1, K), np.uint32)
    j = cross[0] if cross else 1
    codes[0, j] = (1 << bits) - 1
    x = np.zeros((1, K), np.float16)
    x[0, j] = 1.0
    Wq = q4synth.pack_codes(codes, bits)
    want = 2.0 ** -4 * ((1 << bits) - 1) - 0.5
    for mut in ((9, 10) if cross else (9,)):
        assert oracle.gemvb(Wq, s, b, x, bits, mutant=mut)[0][0, 0] != want, mut


@pytest.mark.parametrize("bits", BITS)
def test_brute_force_exact_rational(bits):
    m = q4synth.qb_matrix(820 + bits, 4, 128, bits)
    x = q4synth.activations(821, 2, 128)
    y, A = oracle.gemvb(m.Wq, m.scales, m.biases, x, bits)
    for mm in range(2):
        for n in range(4):
            tot, mag = Fraction(0), Fraction(0)
            for k in range(128):
                w = Fraction(float(m.scales[n, k // 64])) * int(m.codes[n, k]) + Fraction(float(m.biases[n, k // 64]))
                t = w * Fraction(float(x[mm, k]))
                tot += t
                mag += abs(t)
            assert abs(y[mm, n] - float(tot)) <= 1e-15 * float(mag)
            assert abs(A[mm, n] - float(mag)) <= 1e-15 * float(mag)
