"""GPU parity of q4_gemv8 (8-bit codes, same fused-dequant design) against the
fp64 oracle (oracle.gemv8), through the C ABI: shapes across every M with
ragged tails, exact zero rows, general scales and biases, and the
Qwen3-0.6B-shaped lm_head on sampled rows."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


def run8(m, x):
    M, K = x.shape
    y = torch.full((M, m.N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv8(torch_dev(m.Wq), torch_dev(m.scales), torch_dev(m.biases), torch_dev(x), y, M, m.N, K)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 64), (9, 640), (33, 1024), (1000, 2560), (130, 9728), (77, 768)])
def test_shapes_and_batch(M, N, K):
    seed = 5000 + 31 * N + K + 7 * M
    m = q4synth.q8_matrix(seed, N, K)
    x = q4synth.activations(seed + 1, M, K)
    y = run8(m, x)
    y_ref, A = oracle.gemv8(m.Wq, m.scales, m.biases, x)
    assert_parity(y, y_ref, A, what=f"q8 M={M} N={N} K={K}")


def test_zero_rows_are_exact_zero():
    m = q4synth.q8_matrix(51, 64, 1024)
    m.Wq[::3] = 0x80808080
    m.biases[::3] = (-128.0 * m.scales[::3].astype(np.float64)).astype(np.float16)
    y = run8(m, q4synth.activations(52, 2, 1024))
    assert np.all(y[:, ::3] == 0.0)


def test_general_scales_and_biases():
    g = np.random.default_rng(53)
    N, K = 300, 1536
    Wq = g.integers(0, 2**32, size=(N, K // 4), dtype=np.uint32)
    s = (g.standard_normal((N, K // 64)) * 0.003).astype(np.float16)
    b = (g.standard_normal((N, K // 64)) * 0.2).astype(np.float16)
    m = q4synth.Q8Matrix(Wq, s, b)
    for M in (1, 4):
        x = g.standard_normal((M, K)).astype(np.float16)
        y = run8(m, x)
        y_ref, A = oracle.gemv8(Wq, s, b, x)
        assert_parity(y, y_ref, A, what=f"q8 general s,b M={M}")


def test_deterministic_bits():
    m = q4synth.q8_matrix(54, 2000, 2048)
    x = q4synth.activations(55, 3, 2048)
    assert np.array_equal(run8(m, x).view(np.uint32), run8(m, x).view(np.uint32))


def test_full_size_lm_head_sampled_rows():
    shape = q4synth.QWEN3_0P6B
    m = q4synth.q8_matrix(56, shape.vocab, shape.hidden)
    x = q4synth.activations(57, 1, shape.hidden)
    y = run8(m, x)
    rows = np.unique(np.concatenate([np.arange(64), shape.vocab - 1 - np.arange(64),
                                     np.random.default_rng(58).integers(0, shape.vocab, 1024)]))
    y_ref, A = oracle.gemv8(m.Wq, m.scales, m.biases, x, rows=rows)
    assert_parity(y[:, rows], y_ref, A, what="q8 lm_head sampled")
