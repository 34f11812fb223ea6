"""GPU parity of the GEMV for 2-, 3-, 5- and 6-bit codes (q4_gemv_bits, M = 1)
against the fp64 oracle: every element of ragged shapes (a last tile with an
odd row count whose code block is not a 16-byte multiple), every code at the
positions where it crosses a word boundary, exactly-zero rows, and 4/8-bit
calls that must equal q4_gemv / q4_gemv8 bit for bit."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu
WIDTHS = (2, 3, 5, 6)


def run(m, x, bits):
    N, K = m.Wq.shape[0], x.shape[1]
    y = torch.full((1, N), float("nan"), device="cuda")
    q4.q4_gemv_bits(torch_dev(m.Wq), torch_dev(m.scales), torch_dev(m.biases), torch_dev(x), y, 1, N, K, bits)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("N,K", [(300, 320), (77, 1024), (1000, 2048)])
def test_every_element(bits, N, K):
    m = q4synth.qb_matrix(900 + bits + K, N, K, bits)
    x = q4synth.activations(901 + bits, 1, K)
    y = run(m, x, bits)
    y_ref, A = oracle.gemvb(m.Wq, m.scales, m.biases, x, bits)
    assert_parity(y, y_ref, A, what=f"{bits}-bit N={N} K={K}")


@pytest.mark.parametrize("bits", WIDTHS)
def test_every_code_at_crossing_positions(bits):
    K = 128
    cross = [k for k in range(K) if (bits * k) % 32 + bits > 32]
    positions = sorted(set(cross[:6] + [0, 1, 31, 64, K - 1]))
    rows = [(c, j) for j in positions for c in range(1 << bits)]
    codes = np.zeros((len(rows), K), np.uint32)
    for i, (c, j) in enumerate(rows):
        codes[i, j] = c
    s = np.full((len(rows), K // 64), 2.0 ** -4, np.float16)
    b = np.full((len(rows), K // 64), -0.5, np.float16)
    m = q4synth.QbMatrix(q4synth.pack_codes(codes, bits), s, b, bits, codes)
    for j in positions:
        x = np.zeros((1, K), np.float16)
        x[0, j] = 1.0
        y = run(m, x, bits)[0]
        for i, (c, jj) in enumerate(rows):
            want = (2.0 ** -4 * c - 0.5) if jj == j else -0.5
            assert y[i] == want, (bits, j, jj, c, y[i])


@pytest.mark.parametrize("bits", WIDTHS)
def test_zero_rows_are_exact_zero(bits):
    m = q4synth.qb_matrix(950 + bits, 96, 256, bits)
    mid = 1 << (bits - 1)
    codes = m.codes.copy()
    codes[::3] = mid
    biases = m.biases.copy()
    biases[::3] = (-float(mid) * m.scales[::3].astype(np.float64)).astype(np.float16)
    mz = q4synth.QbMatrix(q4synth.pack_codes(codes, bits), m.scales, biases, bits, codes)
    y = run(mz, q4synth.activations(951, 1, 256), bits)
    assert np.all(y[0, ::3] == 0.0)


def test_four_and_eight_bits_match_their_entry_points():
    N, K = 500, 1024
    x = q4synth.activations(960, 1, K)
    for bits, m, fn in ((4, q4synth.q4_matrix(961, N, K), q4.q4_gemv), (8, q4synth.q8_matrix(962, N, K), q4.q4_gemv8)):
        args = (torch_dev(m.Wq), torch_dev(m.scales), torch_dev(m.biases), torch_dev(x))
        y1 = torch.empty(1, N, device="cuda")
        y2 = torch.empty(1, N, device="cuda")
        fn(*args, y1, 1, N, K)
        q4.q4_gemv_bits(*args, y2, 1, N, K, bits)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), bits


def test_refusals():
    z = torch.zeros(64, dtype=torch.int32, device="cuda")
    h = torch.zeros(64, dtype=torch.float16, device="cuda")
    y = torch.zeros(16, device="cuda")
    for bits, M, name in ((7, 1, "Q4_ERR_INVALID_ARG"), (3, 2, "Q4_ERR_UNSUPPORTED")):
        with pytest.raises(q4.Q4Error) as ei:
            q4.q4_gemv_bits(z, h, h, h, y, M, 8, 64, bits)
        assert ei.value.name == name
