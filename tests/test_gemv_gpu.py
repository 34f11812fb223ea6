"""GPU parity of q4_gemv / q4_gemv_ex against the fp64 oracle, through the C ABI.

Shapes span several tiles and ragged tails, every M the kernel serves, the
edge cases (one group, one row, zero rows, general scale/bias values) and the
full-size lm_head of the Qwen3-0.6B-shaped decode stream on sampled rows."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, dev_q4, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


def run_gemv(m, x):
    M, K = x.shape
    Wq, s, b = dev_q4(m)
    y = torch.full((M, m.N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv(Wq, s, b, torch_dev(x), y, M, m.N, K)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return y.cpu().numpy()


def test_single_gemv_m1_k1024_n3072():
    m = q4synth.q4_matrix(q4synth.BASE_SEED, 3072, 1024)
    x = q4synth.activations(q4synth.BASE_SEED + 1, 1, 1024)
    y = run_gemv(m, x)
    y_ref, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    assert_parity(y, y_ref, A, what="M=1 K=1024 N=3072")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(1, 64), (7, 128), (8, 192), (9, 640), (33, 1024), (1000, 2560),
                                 (515, 3072), (130, 9728), (77, 768)])
def test_shapes_and_batch(M, N, K):
    seed = 1000 + 31 * N + K + 7 * M
    m = q4synth.q4_matrix(seed, N, K)
    x = q4synth.activations(seed + 1, M, K)
    y = run_gemv(m, x)
    y_ref, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    assert_parity(y, y_ref, A, what=f"M={M} N={N} K={K}")


def test_general_scales_and_biases():
    """Scales and biases of both signs and unrelated magnitudes (not b = -8 s)."""
    g = np.random.default_rng(77)
    N, K = 300, 1536
    Wq = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s = (g.standard_normal((N, K // 64)) * 0.05).astype(np.float16)
    b = (g.standard_normal((N, K // 64)) * 0.2).astype(np.float16)
    m = q4synth.Q4Matrix(Wq, s, b)
    for M in (1, 4):
        x = g.standard_normal((M, K)).astype(np.float16)
        y = run_gemv(m, x)
        y_ref, A = oracle.gemv(Wq, s, b, x)
        assert_parity(y, y_ref, A, what=f"general s,b M={M}")


def test_zero_rows_are_exact_zero():
    m = q4synth.q4_matrix(21, 64, 1024)
    m.Wq[::3] = 0x88888888
    m.biases[::3] = (-8.0 * m.scales[::3].astype(np.float64)).astype(np.float16)
    x = q4synth.activations(22, 2, 1024)
    y = run_gemv(m, x)
    assert np.all(y[:, ::3] == 0.0)
    y_ref, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    assert_parity(y, y_ref, A, what="zero rows")


def test_hand_worked_golden_example_exact():
    from test_oracle_pins import load_worked_example
    Wq, s, b, x, expect = load_worked_example()
    y = run_gemv(q4synth.Q4Matrix(Wq, s, b), x)
    for n, (yv, _) in expect.items():
        assert y[0, n] == yv


def test_every_code_and_position():
    """One-hot probes: code c at position j of a 128-wide row, x = e_j."""
    rows = []
    for c in range(16):
        for j in range(0, 128, 9):
            w = np.zeros(16, np.uint32)
            w[j // 8] = c << (4 * (j % 8))
            rows.append((w, j, c))
    Wq = np.stack([r[0] for r in rows])
    s = np.full((len(rows), 2), 2.0 ** -4, np.float16)
    b = np.full((len(rows), 2), -0.5, np.float16)
    m = q4synth.Q4Matrix(Wq, s, b)
    for j in range(0, 128, 9):
        x = np.zeros((1, 128), np.float16)
        x[0, j] = 1.0
        y = run_gemv(m, x)
        for i, (_, jj, c) in enumerate(rows):
            want = (2.0 ** -4 * c - 0.5) if jj == j else -0.5   # code 0 elsewhere: w = b
            assert y[0, i] == want, (j, jj, c)


def test_deterministic_bits():
    m = q4synth.q4_matrix(31, 4096, 2048)
    x = q4synth.activations(32, 4, 2048)
    y1 = run_gemv(m, x)
    y2 = run_gemv(m, x)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_fused_segments_fp16_and_residual():
    K = 1024
    mats = [q4synth.q4_matrix(40 + i, n, K) for i, n in enumerate((2048, 1024, 1000, 24))]
    for M in (1, 4):
        x = q4synth.activations(50 + M, M, K)
        res = q4synth.activations(60 + M, M, 1000)
        dev = [dev_q4(mm) for mm in mats]
        ys = [torch.full((M, mm.N), float("nan"), dtype=torch.float16, device="cuda") for mm in mats]
        r_dev = torch_dev(res)
        segs = [q4.Segment(*dev[i], mats[i].N, y=ys[i], residual=(r_dev if i == 2 else None))
                for i in range(4)]
        q4.q4_gemv_ex(segs, torch_dev(x), M, K, out_dtype=q4.Q4_F16)
        torch.cuda.synchronize()
        for i, mm in enumerate(mats):
            y_ref, A = oracle.gemv(mm.Wq, mm.scales, mm.biases, x)
            if i == 2:
                y_ref = y_ref + res.astype(np.float64)
                A = A + np.abs(res.astype(np.float64))
            assert_parity(ys[i].float().cpu().numpy(), y_ref, A, fp16_out=True, what=f"seg {i} M={M}")


def test_residual_in_place():
    K, N = 2048, 1024
    mm = q4synth.q4_matrix(70, N, K)
    x = q4synth.activations(71, 1, K)
    h = q4synth.activations(72, 1, N)
    hd = torch_dev(h)
    q4.q4_gemv_ex([q4.Segment(*dev_q4(mm), N, y=hd, residual=hd)], torch_dev(x), 1, K, out_dtype=q4.Q4_F16)
    torch.cuda.synchronize()
    y_ref, A = oracle.gemv(mm.Wq, mm.scales, mm.biases, x)
    assert_parity(hd.float().cpu().numpy(), y_ref + h, A + np.abs(h.astype(np.float64)), fp16_out=True)


@pytest.mark.parametrize("M,N,K", [(1, 3072, 1024), (4, 8192, 3072), (2, 100, 640), (1, 9728, 2560)])
def test_glu_epilogue(M, N, K):
    g = q4synth.q4_matrix(80 + N, N, K)
    u = q4synth.q4_matrix(81 + N, N, K)
    x = q4synth.activations(82, M, K)
    act = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    q4.q4_gemv_ex([q4.Segment(*dev_q4(g), N, y=act), q4.Segment(*dev_q4(u), N)], torch_dev(x), M, K,
                  out_dtype=q4.Q4_F16, mode=q4.Q4_GEMV_GLU)
    torch.cuda.synchronize()
    gv, Ag = oracle.gemv(g.Wq, g.scales, g.biases, x)
    uv, Au = oracle.gemv(u.Wq, u.scales, u.biases, x)
    ref = oracle.silu(gv) * uv
    # error propagation: |d act| <= |silu'(g)| |u| dg + |silu(g)| du, |silu'| < 1.1
    A = 1.1 * np.abs(uv) * Ag + np.abs(oracle.silu(gv)) * Au
    assert_parity(act.float().cpu().numpy(), ref, A, fp16_out=True, what="GLU")


def test_full_size_lm_head_sampled_rows():
    """Qwen3-0.6B-shaped lm_head (151936 x 1024), checked on sampled rows."""
    shape = q4synth.QWEN3_0P6B
    lm = q4synth.q4_matrix(q4synth.BASE_SEED + 16 * shape.n_layers, shape.vocab, shape.hidden)
    x = q4synth.activations(q4synth.BASE_SEED + 999, 1, shape.hidden)
    y = run_gemv(lm, x)
    rows = np.unique(np.concatenate([np.arange(64), shape.vocab - 1 - np.arange(64),
                                     np.random.default_rng(5).integers(0, shape.vocab, 1024)]))
    y_ref, A = oracle.gemv(lm.Wq, lm.scales, lm.biases, x, rows=rows)
    assert_parity(y[:, rows], y_ref, A, what="lm_head sampled")


@pytest.mark.parametrize("M,K,gamma", [(1, 1024, False), (1, 3072, True), (4, 2560, True), (8, 640, False)])
def test_fused_rmsnorm_prologue(M, K, gamma):
    N = 700
    mm = q4synth.q4_matrix(90 + K, N, K)
    x = (q4synth.activations(91 + K, M, K).astype(np.float32) * 3).astype(np.float16)
    gw = (np.random.default_rng(K).random(K) + 0.5).astype(np.float16) if gamma else None
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv_ex([q4.Segment(*dev_q4(mm), N, y=y)], torch_dev(x), M, K, rmsnorm=True,
                  norm_weight=None if gw is None else torch_dev(gw), norm_eps=1e-5)
    torch.cuda.synchronize()
    y_ref, A = oracle.gemv(mm.Wq, mm.scales, mm.biases, oracle.rmsnorm(x, gw, eps=1e-5))
    assert_parity(y.cpu().numpy(), y_ref, A, what="rmsnorm prologue")


@pytest.mark.parametrize("M", [1, 3])
def test_largest_k_in_one_launch(M):
    """K = 16384: x and two weight stages fill one CTA's shared memory at M = 1;
    M = 3 runs as launches of 2 and 1 rows (each streaming the weights)."""
    N, K = 37, 16384
    m = q4synth.q4_matrix(555, N, K)
    x = q4synth.activations(556, M, K)
    y = run_gemv(m, x)
    y_ref, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    assert_parity(y, y_ref, A, what=f"K={K} M={M}")


def test_k_beyond_shared_memory_is_refused():
    N, K = 8, 32768
    Wq = torch.zeros(N, K // 8, dtype=torch.int32, device="cuda")
    s = torch.zeros(N, K // 64, dtype=torch.float16, device="cuda")
    x = torch.zeros(1, K, dtype=torch.float16, device="cuda")
    y = torch.zeros(1, N, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.q4_gemv(Wq, s, s, x, y, 1, N, K)
    assert ei.value.name == "Q4_ERR_UNSUPPORTED"
    assert q4.q4_device_status() == 0


def test_early_weights_flag_chain():
    """Q4_GEMV_EARLY_WEIGHTS: a chain of launches on one stream where each
    reads the previous one's output (x, and the residual in place) gives the
    same bits as the same chain launched without the flag -- the weights
    stream early, the activations still wait for the kernel before."""
    K, N = 1024, 1024
    mats = [q4synth.q4_matrix(90 + i, N, K) for i in range(6)]
    dev = [dev_q4(mm) for mm in mats]
    x0 = q4synth.activations(96, 1, K)
    outs = []
    for flags in (0, q4.Q4_GEMV_EARLY_WEIGHTS):
        h = torch_dev(x0).clone()
        t = torch.empty(1, N, dtype=torch.float16, device="cuda")
        for i in range(6):
            # t = W_i h; then h += W_i' t (residual in place)
            q4.q4_gemv_ex([q4.Segment(*dev[i], N, y=t)], h, 1, K, out_dtype=q4.Q4_F16, flags=flags)
            q4.q4_gemv_ex([q4.Segment(*dev[(i + 3) % 6], N, y=h, residual=h)], t, 1, K, out_dtype=q4.Q4_F16,
                          flags=flags)
        torch.cuda.synchronize()
        assert q4.q4_device_status() == 0
        outs.append(h.cpu().numpy().copy())
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    # and the first link against the oracle
    t = torch.empty(1, N, dtype=torch.float16, device="cuda")
    q4.q4_gemv_ex([q4.Segment(*dev[0], N, y=t)], torch_dev(x0), 1, K, out_dtype=q4.Q4_F16,
                  flags=q4.Q4_GEMV_EARLY_WEIGHTS)
    torch.cuda.synchronize()
    y_ref, A = oracle.gemv(mats[0].Wq, mats[0].scales, mats[0].biases, x0)
    assert_parity(t.float().cpu().numpy(), y_ref, A, fp16_out=True, what="early weights")
