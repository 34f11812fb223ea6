"""The seeded input generators follow their stated recipe and the workload
shapes are the configurations' shapes (CPU only).

The generators are the one module the tests, the benchmark and the oracle
share, so a slip in them would feed both sides the same wrong inputs and no
parity test could see it.  Checked here: the decode and MoE shapes against
the configurations (layer widths, layer counts, the weight totals they
imply), codes uniform over their range and laid out as the storage format
says (read back bit by bit), scale = fp16(|N(0, 0.02)| / ((2^b - 1) / 2)),
bias = -2^(b-1) * scale exactly, activations N(0, 1) in fp16, and per-tensor
seeding (a matrix regenerates alone from its seed)."""
import numpy as np
import pytest

import q4synth

stats = pytest.importorskip("scipy.stats")


# ------------------------------------------------------------------ shapes ---

def test_qwen3_0p6b_shape():
    s = q4synth.QWEN3_0P6B
    assert (s.n_layers, s.hidden, s.vocab) == (28, 1024, 151936)
    assert s.layer_linears() == [("q", 2048, 1024), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 1024, 2048),
                                 ("gate", 3072, 1024), ("up", 3072, 1024), ("down", 1024, 3072)]
    assert s.weights_per_step() == 595_984_384
    assert s.weight_bytes_per_step() == 335_241_216  # 0.5 B per code + 4 B per group of 64


def test_llama32_3b_and_qwen3_4b_shapes():
    l3 = q4synth.LLAMA32_3B
    assert (l3.n_layers, l3.hidden, l3.vocab) == (28, 3072, 128256)
    assert l3.layer_linears() == [("q", 3072, 3072), ("k", 1024, 3072), ("v", 1024, 3072), ("o", 3072, 3072),
                                  ("gate", 8192, 3072), ("up", 8192, 3072), ("down", 3072, 8192)]
    assert l3.weights_per_step() == 3_212_574_720
    q4b = q4synth.QWEN3_4B
    assert (q4b.n_layers, q4b.hidden, q4b.vocab) == (36, 2560, 151936)
    assert q4b.layer_linears() == [("q", 4096, 2560), ("k", 1024, 2560), ("v", 1024, 2560), ("o", 2560, 4096),
                                   ("gate", 9728, 2560), ("up", 9728, 2560), ("down", 2560, 9728)]
    assert q4b.weights_per_step() == 4_022_272_000


def test_moe_layer_shape():
    m = q4synth.QWEN3_30B_A3B_MOE
    assert (m.hidden, m.experts, m.ffn, m.topk) == (2048, 128, 768, 8)
    weights = m.experts * (2 * m.ffn * m.hidden + m.hidden * m.ffn)
    assert weights // 2 + weights // 64 * 4 == 339_738_624


# ------------------------------------------------------------ 4-bit codes ---

def nibbles(Wq):
    """Codes [.., K] read back from the words: code k in bits 4(k%8).. of word k/8."""
    w = Wq.astype(np.uint64)
    c = np.stack([(w >> (4 * j)) & 15 for j in range(8)], axis=-1)
    return c.reshape(*Wq.shape[:-1], Wq.shape[-1] * 8)


def uniform_ok(codes, n_values):
    counts = np.bincount(codes.ravel().astype(np.int64), minlength=n_values)
    assert counts.size == n_values
    expected = codes.size / n_values
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    return stats.chi2.sf(chi2, n_values - 1) > 1e-6


def half_normal_scale_ok(scales, divisor):
    v = scales.astype(np.float64) * divisor  # ~ |N(0, 0.02)|
    n = v.size
    mean = 0.02 * np.sqrt(2 / np.pi)
    sd = 0.02 * np.sqrt(1 - 2 / np.pi)
    rms = float(np.sqrt((v ** 2).mean()))
    return abs(v.mean() - mean) < 6 * sd / np.sqrt(n) and abs(rms - 0.02) < 0.02 * 6 * np.sqrt(2 / n)


def test_q4_matrix_recipe():
    m = q4synth.q4_matrix(7001, 512, 1024)
    assert m.Wq.dtype == np.uint32 and m.Wq.shape == (512, 128)
    assert m.scales.dtype == np.float16 and m.scales.shape == (512, 16) and m.biases.shape == (512, 16)
    c = nibbles(m.Wq)
    assert c.shape == (512, 1024) and c.max() == 15 and c.min() == 0
    assert uniform_ok(c, 16)
    # neighbouring codes are independent: pairs (code k, code k+1) uniform over 256
    assert uniform_ok(c[:, 0::2] * 16 + c[:, 1::2], 256)
    assert np.all(m.scales >= 0) and np.all(np.isfinite(m.scales.astype(np.float64)))
    assert half_normal_scale_ok(m.scales, 7.5)
    assert np.array_equal(m.biases.astype(np.float64), -8.0 * m.scales.astype(np.float64))


def test_expert_stack_recipe():
    m = q4synth.q4_matrix(7002, 64, 256, experts=8)
    assert m.Wq.shape == (8, 64, 32) and m.scales.shape == (8, 64, 4)
    assert uniform_ok(nibbles(m.Wq), 16)
    assert np.array_equal(m.biases.astype(np.float64), -8.0 * m.scales.astype(np.float64))


def test_activations_and_router_logits():
    for x in (q4synth.activations(7003, 64, 4096), q4synth.router_logits(7004, 2048, 128)):
        assert x.dtype == np.float16
        v = x.astype(np.float64)
        n = v.size
        assert abs(v.mean()) < 6 / np.sqrt(n)
        assert abs(v.std() - 1.0) < 6 * np.sqrt(0.5 / n)
        assert stats.kstest(v.ravel()[:20000], "norm").pvalue > 1e-6


def test_seeding_regenerates_single_tensors():
    a, b = q4synth.q4_matrix(9, 32, 128), q4synth.q4_matrix(9, 32, 128)
    assert np.array_equal(a.Wq, b.Wq) and np.array_equal(a.scales, b.scales)
    assert not np.array_equal(a.Wq, q4synth.q4_matrix(10, 32, 128).Wq)
    shape = q4synth.tiny_decode_shape(n_layers=2)
    layers, lm = q4synth.decode_weights(shape)
    for l, d in enumerate(layers):
        for j, (nm, N, K) in enumerate(shape.layer_linears()):
            alone = q4synth.q4_matrix(q4synth.BASE_SEED + 16 * l + j, N, K)
            assert np.array_equal(d[nm].Wq, alone.Wq) and np.array_equal(d[nm].scales, alone.scales)
    assert np.array_equal(lm.Wq, q4synth.q4_matrix(q4synth.BASE_SEED + 32, shape.vocab, shape.hidden).Wq)


def test_k_must_be_a_group_multiple():
    for make in (lambda: q4synth.q4_matrix(1, 8, 100), lambda: q4synth.q8_matrix(1, 8, 100),
                 lambda: q4synth.qb_matrix(1, 8, 100, 3)):
        with pytest.raises(ValueError):
            make()


# ----------------------------------------------------- 8-bit, b-bit codes ---

def test_q8_matrix_recipe():
    m = q4synth.q8_matrix(7005, 256, 1024)
    assert m.Wq.shape == (256, 256)
    w = m.Wq.astype(np.uint64)
    c = np.stack([(w >> (8 * j)) & 255 for j in range(4)], axis=-1).reshape(256, 1024)
    assert uniform_ok(c, 256)
    assert half_normal_scale_ok(m.scales, 127.5)
    assert np.array_equal(m.biases.astype(np.float64), -128.0 * m.scales.astype(np.float64))


@pytest.mark.parametrize("bits", [2, 3, 5, 6])
def test_qb_matrix_recipe_and_bit_stream(bits):
    m = q4synth.qb_matrix(7006 + bits, 128, 640, bits)
    assert m.Wq.shape == (128, 640 * bits // 32) and m.codes.shape == (128, 640)
    assert uniform_ok(m.codes, 1 << bits)
    assert half_normal_scale_ok(m.scales, (2 ** bits - 1) / 2)
    assert np.array_equal(m.biases.astype(np.float64), -(2.0 ** (bits - 1)) * m.scales.astype(np.float64))
    # the packed words hold code k at bits b*k .. b*k+b-1 of the row's stream
    for n in (0, 77, 127):
        row = [int(x) for x in m.Wq[n]]
        stream = sum(w << (32 * i) for i, w in enumerate(row))
        for k in range(640):
            assert (stream >> (bits * k)) & ((1 << bits) - 1) == int(m.codes[n, k]), (bits, n, k)


def test_pack_codes_hand_example():
    # 3-bit codes 1..7,0 repeated: the first word holds codes 0..9 whole and the
    # low two bits of code 10
    codes = np.array([[1, 2, 3, 4, 5, 6, 7, 0] * 4], dtype=np.uint32)
    w = q4synth.pack_codes(codes, 3)
    expect0 = 0
    for k in range(11):
        expect0 |= (int(codes[0, k]) << (3 * k)) & 0xFFFFFFFF
    assert int(w[0, 0]) == expect0
    assert int(w[0, 1]) & 1 == (int(codes[0, 10]) >> 2) & 1
