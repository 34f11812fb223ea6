"""Pins for the CPU oracle: checks against facts fixed outside the oracle itself
(hand-worked examples, exact rational arithmetic, closed forms, invariants,
an independent library routine), chosen so a plausible mistake in the oracle
fails at least one of them (``test_planted_mistakes_are_caught``)."""
from fractions import Fraction
import os

import numpy as np
import pytest

import oracle
import q4synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def h(v):
    """fp16 bit pattern of an exactly representable value."""
    return int(np.array([v], np.float16).view(np.uint16)[0])


def unpack_codes(Wq):
    """Independent unpacking for the pins: code k of a row sits in word k//8,
    bits 4*(k%8)..+3 (lowest nibble first)."""
    N, W = Wq.shape
    codes = np.zeros((N, W * 8), np.int64)
    for i in range(8):
        codes[:, i::8] = (Wq.astype(np.int64) >> (4 * i)) & 0xF
    return codes


def exact_gemv(Wq, s, b, x):
    """Exact rational y[n] = sum_k (s q + b) x, fractions only."""
    codes = unpack_codes(Wq)
    N, K = codes.shape
    sf = [[Fraction(float(v)) for v in row] for row in s.astype(np.float64)]
    bf = [[Fraction(float(v)) for v in row] for row in b.astype(np.float64)]
    xf = [Fraction(float(v)) for v in x.astype(np.float64).ravel()]
    out = []
    for n in range(N):
        acc = Fraction(0)
        for k in range(K):
            g = k // 64
            acc += (sf[n][g] * int(codes[n, k]) + bf[n][g]) * xf[k]
        out.append(acc)
    return out


def one_group(words, s_val, b_val):
    Wq = np.array([words], np.uint32)
    s = np.full((1, len(words) // 8), s_val, np.float16)
    b = np.full((1, len(words) // 8), b_val, np.float16)
    return Wq, s, b


# ------------------------------------------------------------ fp16 decode ---

def test_half_to_double_known_patterns():
    cases = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
             0x03FF: 1023 * 2.0 ** -24, 0x0400: 2.0 ** -14, 0x3555: 0.333251953125,
             0x8000: -0.0, 0x7C00: float("inf"), 0xFC00: float("-inf")}
    for bits, v in cases.items():
        assert oracle.half_to_double(bits) == v, hex(bits)


def test_half_to_double_matches_numpy_everywhere():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(v)) for v in bits])
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


# ------------------------------------------------------------- code map -----

def code_probe(code, pos, mutant=0, s_val=2.0 ** -4, b_val=-0.5):
    """One group with code ``code`` at position ``pos`` (others 0), x = e_pos."""
    words = [0] * 8
    words[pos // 8] = code << (4 * (pos % 8))
    Wq, s, b = one_group(words, s_val, b_val)
    x = np.zeros((1, 64), np.float16)
    x[0, pos] = 1.0
    y, A = oracle.gemv(Wq, s, b, x, mutant=mutant)
    return y[0, 0], A[0, 0]


def test_every_code_maps_exactly():
    for code in range(16):
        for pos in range(64):
            y, A = code_probe(code, pos)
            want = 2.0 ** -4 * code - 0.5
            assert y == want and A == abs(want), (code, pos)


def test_nibble_order_low_first():
    words = [0x76543210, 0xFEDCBA98] * 4
    Wq, s, b = one_group(words, 1.0, 0.0)
    for k in range(64):
        x = np.zeros((1, 64), np.float16)
        x[0, k] = 1.0
        y, _ = oracle.gemv(Wq, s, b, x)
        assert y[0, 0] == k % 16, k


def load_worked_example():
    rows, scales, biases, x, expect = {}, {}, {}, {}, {}
    K = N = None
    with open(os.path.join(GOLDEN, "q4_worked_example.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "K":
                K = int(t[1])
            elif t[0] == "N":
                N = int(t[1])
            elif t[0] == "row" and t[2] == "words":
                rows[int(t[1])] = [int(v, 16) for v in t[3:]]
            elif t[0] == "row" and t[2] == "scales":
                scales[int(t[1])] = [int(v, 16) for v in t[3:5]]
                biases[int(t[1])] = [int(v, 16) for v in t[6:8]]
            elif t[0] == "x":
                for kv in t[1:]:
                    k, v = kv.split(":")
                    x[int(k)] = int(v, 16)
            elif t[0] == "expect":
                expect[int(t[1])] = (float(t[2]), float(t[3]))
    Wq = np.array([rows[n] * (K // 8 // len(rows[n])) for n in range(N)], np.uint32)
    s = np.array([scales[n] for n in range(N)], np.uint16).view(np.float16)
    b = np.array([biases[n] for n in range(N)], np.uint16).view(np.float16)
    xv = np.zeros((1, K), np.uint16)
    for k, v in x.items():
        xv[0, k] = v
    return Wq, s, b, xv.view(np.float16), expect


def test_hand_worked_example():
    Wq, s, b, x, expect = load_worked_example()
    y, A = oracle.gemv(Wq, s, b, x)
    for n, (yv, av) in expect.items():
        assert y[0, n] == yv and A[0, n] == av, n


# --------------------------------------------------- closed form, brute force

@pytest.mark.parametrize("K", [64, 1024, 9728])
def test_all_ones_closed_form(K):
    """x = 1: y_n = sum_g (s_g * sum_{k in g} q_k + 64 b_g), exact in fp64."""
    m = q4synth.q4_matrix(7 + K, 6, K)
    codes = unpack_codes(m.Wq)
    x = np.ones((1, K), np.float16)
    y, _ = oracle.gemv(m.Wq, m.scales, m.biases, x)
    for n in range(6):
        want = Fraction(0)
        for g in range(K // 64):
            qs = int(codes[n, 64 * g:64 * g + 64].sum())
            want += Fraction(float(m.scales[n, g])) * qs + 64 * Fraction(float(m.biases[n, g]))
        assert y[0, n] == float(want), n


@pytest.mark.parametrize("K,N", [(64, 16), (128, 9)])
def test_brute_force_exact_rationals(K, N):
    m = q4synth.q4_matrix(100 + K, N, K)
    x = q4synth.activations(200 + K, 1, K)
    y, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    exact = exact_gemv(m.Wq, m.scales, m.biases, x)
    for n in range(N):
        assert abs(y[0, n] - float(exact[n])) <= 1e-15 * max(A[0, n], 1e-300)


def test_brute_force_general_scales_and_biases():
    """Arbitrary fp16 scales/biases of both signs, not only b = -8 s."""
    g = np.random.default_rng(5)
    N, K = 7, 128
    Wq = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s = g.standard_normal((N, 2)).astype(np.float16)
    b = g.standard_normal((N, 2)).astype(np.float16)
    x = g.standard_normal((1, K)).astype(np.float16)
    y, A = oracle.gemv(Wq, s, b, x)
    exact = exact_gemv(Wq, s, b, x)
    for n in range(N):
        assert abs(y[0, n] - float(exact[n])) <= 1e-15 * A[0, n]


# ------------------------------------------------------------- invariants ---

def test_zero_row_exact():
    m = q4synth.q4_matrix(11, 4, 256)
    Wq = np.full_like(m.Wq, 0x88888888)
    b = (-8.0 * m.scales.astype(np.float64)).astype(np.float16)
    x = q4synth.activations(12, 2, 256)
    y, A = oracle.gemv(Wq, m.scales, b, x)
    assert np.all(y == 0.0) and np.all(A == 0.0)


def test_negating_x_negates_y_exactly():
    m = q4synth.q4_matrix(13, 10, 512)
    x = q4synth.activations(14, 1, 512)
    y1, A1 = oracle.gemv(m.Wq, m.scales, m.biases, x)
    y2, A2 = oracle.gemv(m.Wq, m.scales, m.biases, -x)
    assert np.array_equal(y1, -y2) and np.array_equal(A1, A2)


def test_bias_shift_adds_group_sum():
    m = q4synth.q4_matrix(15, 3, 192)
    x = q4synth.activations(16, 1, 192)
    y0, _ = oracle.gemv(m.Wq, m.scales, m.biases, x)
    b2 = m.biases.copy()
    b2[1, 2] = np.float16(float(b2[1, 2]) + 0.25)
    delta = float(b2[1, 2]) - float(m.biases[1, 2])   # the shift actually stored
    assert delta != 0.0
    y1, _ = oracle.gemv(m.Wq, m.scales, b2, x)
    xs = x.astype(np.float64)[0, 128:192].sum()
    assert abs((y1[0, 1] - y0[0, 1]) - delta * xs) <= 1e-12 * (1 + abs(y0[0, 1]))
    assert y1[0, 0] == y0[0, 0] and y1[0, 2] == y0[0, 2]


def test_rows_subset_and_batch_agree():
    m = q4synth.q4_matrix(17, 40, 320)
    x = q4synth.activations(18, 3, 320)
    y, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    rows = np.array([39, 0, 17, 17, 5])
    ys, As = oracle.gemv(m.Wq, m.scales, m.biases, x, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(As, A[:, rows])
    for mm in range(3):
        y1, _ = oracle.gemv(m.Wq, m.scales, m.biases, x[mm:mm + 1])
        assert np.array_equal(y1[0], y[mm])


def test_threads_do_not_change_results():
    m = q4synth.q4_matrix(19, 64, 1024)
    x = q4synth.activations(20, 1, 1024)
    y1, _ = oracle.gemv(m.Wq, m.scales, m.biases, x, nthreads=1)
    y4, _ = oracle.gemv(m.Wq, m.scales, m.biases, x, nthreads=4)
    assert np.array_equal(y1, y4)


# ----------------------------------------------------- planted mistakes -----

def _pins_pass(mutant):
    """Run a subset of the pins against oracle variant ``mutant``."""
    ok = True
    for code in (0, 3, 15):
        for pos in (0, 5, 63):
            y, _ = code_probe(code, pos, mutant=mutant)
            ok &= (y == 2.0 ** -4 * code - 0.5)
    Wq, s, b, x, expect = load_worked_example()
    y, A = oracle.gemv(Wq, s, b, x, mutant=mutant)
    ok &= all(y[0, n] == e[0] and A[0, n] == e[1] for n, e in expect.items())
    return bool(ok)


def test_real_oracle_passes_pin_subset():
    assert _pins_pass(0)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_planted_mistakes_are_caught(mutant):
    """1: nibble order reversed, 2: bias dropped, 3: group 32 instead of 64,
    4: bias sign flipped, 5: x indexed by the row (transposed operand)."""
    assert not _pins_pass(mutant)


# --------------------------------------------------- fp16 store, SiLU -------

def test_fp16_rounding_is_rne_from_double():
    one = 1.0
    assert oracle.fp16(one + 2.0 ** -11) == 1.0                      # tie -> even
    assert oracle.fp16(one + 3 * 2.0 ** -11) == one + 2.0 ** -9        # tie -> even (up)
    assert oracle.fp16(one + 2.0 ** -11 + 2.0 ** -40) == one + 2.0 ** -10  # no double rounding
    assert oracle.fp16(65520.0) == np.inf                              # overflow threshold
    assert oracle.fp16(2.0 ** -25) == 0.0 and oracle.fp16(2.0 ** -25 + 2.0 ** -40) == 2.0 ** -24


def test_silu_invariants():
    x = np.linspace(-30, 30, 601)
    s = oracle.silu(x)
    assert oracle.silu(0.0) == 0.0
    assert np.allclose(s - oracle.silu(-x), x, rtol=0, atol=1e-12)   # x*sig(x) + x*sig(-x)... = x
    assert np.all(s[x > 0] > 0) and np.all(s[x < 0] < 0)
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12 and abs(oracle.silu(-40.0)) < 1e-15
    assert s.min() > -0.2785 and s.min() < -0.2784                    # global minimum of SiLU


def test_ulp16():
    assert oracle.ulp16(1.0) == 2.0 ** -10
    assert oracle.ulp16(1.5) == 2.0 ** -10
    assert oracle.ulp16(0.0) == 2.0 ** -24
    assert oracle.ulp16(65504.0) == 32.0
