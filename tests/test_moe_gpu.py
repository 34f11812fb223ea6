"""GPU parity of the MoE prefill pieces against the oracle: routing (bit-exact
ids, offsets, permutation), gather (exact), combine (fp32 tolerance)."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


def gpu_route(logits, topk):
    T, E = logits.shape
    R = T * topk
    dev = lambda *s, dt=torch.int32: torch.full(s, -7, dtype=dt, device="cuda")
    ids, w = dev(T, topk), torch.full((T, topk), float("nan"), device="cuda")
    off, tok, exp, pos = dev(E + 1), dev(R), dev(R), dev(T, topk)
    nws = q4.q4_moe_route_workspace_bytes(T, E, topk)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    q4.q4_moe_route(torch_dev(logits), T, E, topk, ids, w, off, tok, exp, pos, ws, nws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in dict(ids=ids, weights=w, offsets=off, token_of=tok, expert_of=exp,
                                                 pos=pos).items()}


def check_route(logits, topk):
    g = gpu_route(logits, topk)
    r = oracle.moe_route(logits, topk)
    for k in ("ids", "offsets", "token_of", "expert_of", "pos"):
        assert np.array_equal(g[k], r[k]), k
    assert np.max(np.abs(g["weights"] - r["weights"])) <= 1e-6
    return g, r


def test_route_hand_worked_fixture():
    from test_oracle_stream_pins import load_routing_fixture
    fx = load_routing_fixture()
    g, _ = check_route(fx["logits"], fx["topk"])
    assert np.array_equal(g["ids"], fx["ids"]) and np.array_equal(g["pos"], fx["pos"])


@pytest.mark.parametrize("T", [1, 31, 128, 512, 2048])
def test_route_qwen3_30b_a3b_shape(T):
    check_route(q4synth.router_logits(q4synth.BASE_SEED + T, T, 128), 8)


@pytest.mark.parametrize("T,E,k", [(100, 16, 4), (33, 8, 8), (65, 256, 1), (7, 3, 2)])
def test_route_ties_and_odd_shapes(T, E, k):
    g = np.random.default_rng(T + E)
    logits = (g.integers(-2, 3, size=(T, E)) * 0.5).astype(np.float16)
    logits[0, :] = 0
    logits[-1, ::2] = -0.0
    check_route(logits, k)


def test_gather_exact():
    T, K, topk = 64, 2048, 8
    r = oracle.moe_route(q4synth.router_logits(5, T, 128), topk)
    X = q4synth.activations(6, T, K)
    Xs = torch.full((T * topk, K), float("nan"), dtype=torch.float16, device="cuda")
    q4.q4_moe_gather(torch_dev(X), T, K, torch_dev(r["token_of"]), T * topk, Xs)
    torch.cuda.synchronize()
    assert np.array_equal(Xs.cpu().numpy().view(np.uint16), X[r["token_of"]].view(np.uint16))


@pytest.mark.parametrize("ydt,odt", [(0, 0), (1, 1), (1, 0), (0, 1)])
def test_combine(ydt, odt):
    T, N, topk = 96, 2048, 8
    r = oracle.moe_route(q4synth.router_logits(7, T, 128), topk)
    Y = np.random.default_rng(8).standard_normal((T * topk, N))
    Y = Y.astype(np.float16) if ydt else Y.astype(np.float32)
    out = torch.empty(T, N, dtype=torch.float16 if odt else torch.float32, device="cuda")
    w = r["weights"].astype(np.float32)
    q4.q4_moe_combine(torch_dev(Y), ydt, N, torch_dev(r["pos"]), torch_dev(w), T, topk, out, odt)
    torch.cuda.synchronize()
    ref, mag = oracle.moe_combine(Y.astype(np.float64), r["pos"], w.astype(np.float64))
    # fp32 accumulation of 8 terms: relative 1e-6 of the magnitudes, plus the fp16 store
    assert_parity(out.float().cpu().numpy(), ref, mag, fp16_out=bool(odt), what="combine")


@pytest.mark.parametrize("ydt,odt", [(1, 1), (0, 0)])
def test_combine_vector_and_scalar_paths_agree(ydt, odt):
    """N % 8 == 0 with aligned buffers takes the 16-byte path; a misaligned
    output takes the per-element path: same arithmetic, identical bits.  An N
    that is not a multiple of 8 is checked against the oracle."""
    T, N, topk = 40, 1024, 8
    r = oracle.moe_route(q4synth.router_logits(17, T, 64), topk)
    Y = np.random.default_rng(18).standard_normal((T * topk, N))
    Y = Y.astype(np.float16) if ydt else Y.astype(np.float32)
    w = torch_dev(r["weights"].astype(np.float32))
    pos = torch_dev(r["pos"])
    dt = torch.float16 if odt else torch.float32
    a = torch.empty(T, N, dtype=dt, device="cuda")
    big = torch.empty(T * N + 1, dtype=dt, device="cuda")
    b = big[1:]                                   # 2 or 4 bytes off a 16-byte boundary
    q4.q4_moe_combine(torch_dev(Y), ydt, N, pos, w, T, topk, a, odt)
    q4.q4_moe_combine(torch_dev(Y), ydt, N, pos, w, T, topk, b, odt)
    torch.cuda.synchronize()
    assert torch.equal(a.flatten(), b)
    N2 = 100
    Y2 = np.random.default_rng(19).standard_normal((T * topk, N2)).astype(Y.dtype)
    c = torch.empty(T, N2, dtype=dt, device="cuda")
    q4.q4_moe_combine(torch_dev(Y2), ydt, N2, pos, w, T, topk, c, odt)
    torch.cuda.synchronize()
    ref, mag = oracle.moe_combine(Y2.astype(np.float64), r["pos"], r["weights"].astype(np.float64))
    assert_parity(c.float().cpu().numpy(), ref, mag, fp16_out=bool(odt), what="combine N=100")
