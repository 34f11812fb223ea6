"""GPU parity of the clustered decode step (one launch of thread-block
clusters for the layer stack, two grid-wide hand-offs per layer, then the
lm_head GEMV) against the oracle's decode stream.

Tables with Q4_DECODE_CLUSTERED whose widths are multiples of 512 take this
path (q4_decode_path == 3).  Every stage of every layer is checked from the GPU's
own stage input (the tight per-element bound), the end-to-end logits to
relative L2 <= 1e-3; the same input twice gives the same bits; the exchange
tags stay correct over many steps; the per-stage launches (the default)
agree within the bound; the full Qwen3-0.6B-shaped stack matches the oracle
stage by stage on sampled rows and end to end."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import torch_dev
from test_decode_gpu import DevModel, run_every_stage

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu

CLUSTERED = 3
F = q4.Q4_DECODE_CLUSTERED


@pytest.fixture(scope="module")
def small():
    return DevModel(q4synth.tiny_decode_shape(n_layers=3, hidden=512, q=1024, kv=256, ffn=1536, vocab=1000),
                    seed=q4synth.BASE_SEED + 70)


@pytest.fixture(scope="module")
def small_gamma():
    return DevModel(q4synth.tiny_decode_shape(n_layers=2, hidden=1024, q=2048, kv=512, ffn=2560, vocab=777),
                    seed=q4synth.BASE_SEED + 71, gammas=True, eps=1e-5)


def path_of(model, n_layers, flags=F):
    t = model.table(n_layers, 1, flags)
    x = torch_dev(q4synth.activations(5, 1, model.shape.hidden))
    lg = torch.empty(1, model.shape.vocab, device="cuda")
    q4.q4_decode_step(t, x, lg)
    torch.cuda.synchronize()
    path = q4.q4_decode_path(t)
    t.release()
    return path


def test_clustered_path_is_taken(small, small_gamma):
    assert path_of(small, 3) == CLUSTERED
    assert path_of(small_gamma, 2) == CLUSTERED
    assert path_of(small, 3, flags=0) == 1


def test_every_stage_and_end_to_end(small):
    run_every_stage(small, 1, q4synth.BASE_SEED + 800, flags=F)


def test_norm_weights_every_stage_and_end_to_end(small_gamma):
    run_every_stage(small_gamma, 1, q4synth.BASE_SEED + 801, flags=F)


def test_same_input_same_bits_and_stages_agree(small):
    x = q4synth.activations(q4synth.BASE_SEED + 802, 1, small.shape.hidden)
    a = small.step(3, x, flags=F)
    b = small.step(3, x, flags=F)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    s = small.step(3, x)
    rel = np.linalg.norm(a["logits"] - s["logits"]) / np.linalg.norm(s["logits"])
    assert rel <= 1e-3, rel


def test_many_steps_stay_correct(small):
    """Every step writes every exchange with a new tag; 300 replays keep the
    first step's bits and match the oracle."""
    t = small.table(3, 1, flags=F)
    xs = q4synth.activations(q4synth.BASE_SEED + 803, 1, small.shape.hidden)
    x_dev = torch_dev(xs)
    lg = torch.empty(1, small.shape.vocab, device="cuda")
    first = None
    for i in range(300):
        q4.q4_decode_step(t, x_dev, lg)
        if i == 0:
            torch.cuda.synchronize()
            first = lg.cpu().numpy().copy()
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    assert q4.q4_decode_path(t) == CLUSTERED
    last = lg.cpu().numpy()
    t.release()
    assert np.array_equal(first.view(np.uint32), last.view(np.uint32))
    ref, _, _ = oracle.decode_step(small.layers, small.lm, xs)
    assert np.linalg.norm(last - ref) / np.linalg.norm(ref) <= 1e-3


def test_direct_launches_equal_graph(small):
    x = q4synth.activations(q4synth.BASE_SEED + 804, 1, small.shape.hidden)
    a = small.step(2, x, flags=F)
    for fl in (q4.Q4_DECODE_NO_GRAPH, q4.Q4_DECODE_NO_PDL):
        o = small.step(2, x, flags=F | fl)
        for k in a:
            assert np.array_equal(a[k], o[k]), (fl, k)


@pytest.fixture(scope="module")
def qwen06():
    return DevModel(q4synth.QWEN3_0P6B)


def test_qwen3_0p6b_full_size(qwen06):
    """The full Qwen3-0.6B-shaped stream on the clustered step: every stage of
    the last layer on sampled rows, sampled logits, end-to-end logits."""
    from helpers import assert_parity
    from test_decode_gpu import check_layer
    s = qwen06.shape
    x = q4synth.activations(q4synth.BASE_SEED + 778, 1, s.hidden)
    prev = qwen06.step(s.n_layers - 1, x, flags=F)
    out = qwen06.step(s.n_layers, x, flags=F)
    g = np.random.default_rng(4)
    rows = {"qkv": {"q": g.integers(0, s.q, 256), "k": g.integers(0, s.kv, 128), "v": g.integers(0, s.kv, 128)},
            "hidden": np.unique(g.integers(0, s.hidden, 256)), "ffn": np.unique(g.integers(0, s.ffn, 256))}
    check_layer(qwen06.layers[-1], prev["h"].astype(np.float16), out, rows=rows, what="last layer")
    lrows = np.unique(g.integers(0, s.vocab, 2048))
    y_ref, A = oracle.decode_logits(qwen06.lm, out["h"], rows=lrows)
    assert_parity(out["logits"][:, lrows], y_ref, A, what="logits sampled")
    l_ref, _, _ = oracle.decode_step(qwen06.layers, qwen06.lm, x)
    rel = np.linalg.norm(out["logits"] - l_ref) / np.linalg.norm(l_ref)
    assert rel <= 1e-3, rel
