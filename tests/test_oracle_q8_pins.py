"""Pins of the 8-bit-code oracle (oracle.gemv8) against facts fixed outside it.

The 8-bit format (BaseRT §3.3 / §4.1 evaluate Q4 and Q8; the bit layout is
the library's): Wq uint32 [N, K/4], code k in byte k % 4 of word k // 4
(lowest byte first), fp16 scale and bias per 64-group, w = s * q + b.

* every code 0..255 at every position of a group maps exactly;
* the byte order, read with numpy's little-endian byte view;
* the all-ones closed form y = sum_g (s_g * sum q + 64 * b_g), exact;
* brute force in exact rationals for tiny K with scales and biases of both
  signs (independent of the oracle's code extraction: codes from the byte view);
* a zero row (q = 128, b = -128 s) gives exactly 0;
* three planted mistakes (byte order, nibble instead of byte, 32-wide groups)
  each fail one of these pins."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import q4synth


def pack8(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [N, K] -> uint32 words [N, K/4], lowest byte first."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return c.view("<u4").reshape(c.shape[0], c.shape[1] // 4).astype(np.uint32)


def codes_of(Wq: np.ndarray) -> np.ndarray:
    """The inverse of pack8, by numpy's byte view (not the oracle's shifts)."""
    w = np.ascontiguousarray(Wq, dtype="<u4")
    return w.view(np.uint8).reshape(w.shape[0], w.shape[1] * 4)


def test_pack_and_view_are_inverse():
    c = np.random.default_rng(0).integers(0, 256, size=(3, 128), dtype=np.uint8)
    assert np.array_equal(codes_of(pack8(c)), c)


def every_code_every_position(mutant=0):
    """Row c holds code c at all 64 positions; x row p is one-hot at p."""
    K = 64
    codes = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K, axis=1)
    Wq = pack8(codes)
    s = np.ones((256, 1), np.float16)
    b = np.zeros((256, 1), np.float16)
    x = np.eye(K, dtype=np.float16)
    y, _ = oracle.gemv8(Wq, s, b, x, mutant=mutant)
    return np.array_equal(y, np.broadcast_to(np.arange(256, dtype=np.float64), (K, 256)))


def byte_order(mutant=0):
    """Code k = k at position k (k < 64): x one-hot at p must give y = p."""
    codes = np.arange(64, dtype=np.uint8)[None, :]
    y, _ = oracle.gemv8(pack8(codes), np.ones((1, 1), np.float16), np.zeros((1, 1), np.float16),
                        np.eye(64, dtype=np.float16), mutant=mutant)
    return np.array_equal(y[:, 0], np.arange(64, dtype=np.float64))


def all_ones_closed_form(K=256, mutant=0):
    m = q4synth.q8_matrix(7, 5, K)
    y, _ = oracle.gemv8(m.Wq, m.scales, m.biases, np.ones((1, K), np.float16), mutant=mutant)
    q = codes_of(m.Wq).astype(np.int64)
    for n in range(m.N):
        want = Fraction(0)
        for g in range(K // 64):
            want += Fraction(float(m.scales[n, g])) * int(q[n, 64 * g:64 * g + 64].sum()) + \
                64 * Fraction(float(m.biases[n, g]))
        if Fraction(y[0, n]) != want:
            return False
    return True


def test_every_code_at_every_position_maps_exactly():
    assert every_code_every_position()


def test_byte_order_lowest_first():
    assert byte_order()
    row = pack8(np.array([[1, 2, 3, 4, 5, 6, 7, 8] + [0] * 56], np.uint8))[0]
    assert [oracle.code8(row, k) for k in range(8)] == [1, 2, 3, 4, 5, 6, 7, 8]


@pytest.mark.parametrize("K", [64, 256, 1024])
def test_all_ones_closed_form(K):
    assert all_ones_closed_form(K)


@pytest.mark.parametrize("K,N", [(64, 3), (128, 2)])
def test_brute_force_exact_rationals(K, N):
    g = np.random.default_rng(K + N)
    codes = g.integers(0, 256, size=(N, K), dtype=np.uint8)
    s = (g.standard_normal((N, K // 64)) * 0.01).astype(np.float16)
    b = (g.standard_normal((N, K // 64)) * 0.5).astype(np.float16)
    x = g.standard_normal((2, K)).astype(np.float16)
    y, A = oracle.gemv8(pack8(codes), s, b, x)
    for m in range(2):
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                w = Fraction(float(s[n, k // 64])) * int(codes[n, k]) + Fraction(float(b[n, k // 64]))
                exact += w * Fraction(float(x[m, k]))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(A[m, n]) * Fraction(1, 2 ** 50)


def test_zero_row_exact():
    m = q4synth.q8_matrix(9, 4, 512)
    m.Wq[1] = 0x80808080                       # q = 128 everywhere
    m.biases[1] = (-128.0 * m.scales[1].astype(np.float64)).astype(np.float16)
    y, A = oracle.gemv8(m.Wq, m.scales, m.biases, q4synth.activations(10, 3, 512))
    assert np.all(y[:, 1] == 0.0) and np.all(A[:, 1] == 0.0)


def _pins_pass(mutant):
    return every_code_every_position(mutant) and byte_order(mutant) and all_ones_closed_form(256, mutant)


def test_real_oracle_passes_pin_subset():
    assert _pins_pass(0)


@pytest.mark.parametrize("mutant", [6, 7, 8])
def test_planted_mistakes_are_caught(mutant):
    oracle.build(mutant)
    assert not _pins_pass(mutant)
