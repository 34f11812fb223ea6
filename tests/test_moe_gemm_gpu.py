"""GPU parity of the tcgen05 grouped GEMM (q4_moe_gemm) and of the whole MoE
prefill layer (route -> gather -> gate/up GEMM -> down GEMM -> combine)
against the fp64 oracle.

Small cases are compared on every element (experts with 0, 1, 17, 128 and
200 rows: empty experts, ragged token tiles, more than one token tile); the
Qwen3-30B-A3B-shaped layer (128 experts, top-8, hidden 2048, expert FFN 768)
at 128 / 512 / 2048 tokens is compared on sampled rows, and end to end at a
small token count."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, dev_q4, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


def offsets_from_counts(counts):
    off = np.zeros(len(counts) + 1, np.int32)
    off[1:] = np.cumsum(counts)
    return off


def run_gemm(W, X, counts, N, K, mode, out_dtype):
    E = len(counts)
    off = offsets_from_counts(counts)
    R = int(off[-1])
    eids = np.repeat(np.arange(E, dtype=np.int32), counts)
    Y = torch.full((R, N), float("nan"), dtype=torch.float16 if out_dtype == q4.Q4_F16 else torch.float32,
                   device="cuda")
    q4.q4_moe_gemm(*dev_q4(W), torch_dev(X), torch_dev(eids), torch_dev(off), Y, E, N, K, R, mode, out_dtype)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return Y.float().cpu().numpy(), eids


def check_plain(W, X, eids, Y, rows=None, fp16_out=False, what=""):
    rows = np.arange(len(eids)) if rows is None else rows
    for r in rows:
        e = eids[r]
        y_ref, A = oracle.gemv(W.Wq[e], W.scales[e], W.biases[e], X[r:r + 1])
        assert_parity(Y[r:r + 1], y_ref, A, fp16_out=fp16_out, what=f"{what} row {r} expert {e}")


def check_glu(W, X, eids, H, ffn, rows=None, what=""):
    rows = np.arange(len(eids)) if rows is None else rows
    g, Ag, u, Au, act = oracle.moe_gate_up_rows(W, X[rows], eids[rows], ffn)
    A = 1.1 * np.abs(u) * Ag + np.abs(oracle.silu(g)) * Au
    assert_parity(H[rows], act, A, fp16_out=True, what=what)


COUNTS = [0, 1, 17, 128, 200, 0, 3]


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_plain_small_every_element(out_dtype):
    N, K = 256, 192
    W = q4synth.q4_matrix(300, N, K, experts=len(COUNTS))
    X = q4synth.activations(301, sum(COUNTS), K)
    Y, eids = run_gemm(W, X, COUNTS, N, K, q4.Q4_GEMV_PLAIN, out_dtype)
    check_plain(W, X, eids, Y, fp16_out=bool(out_dtype), what="plain")


def test_glu_small_every_element():
    ffn, K = 128, 256
    W = q4synth.q4_matrix(310, 2 * ffn, K, experts=len(COUNTS))
    X = q4synth.activations(311, sum(COUNTS), K)
    H, eids = run_gemm(W, X, COUNTS, ffn, K, q4.Q4_GEMV_GLU, q4.Q4_F16)
    check_glu(W, X, eids, H, ffn, what="glu")


def test_one_expert_one_row():
    N, K = 128, 64
    W = q4synth.q4_matrix(340, N, K, experts=1)
    X = q4synth.activations(341, 1, K)
    Y, eids = run_gemm(W, X, [1], N, K, q4.Q4_GEMV_PLAIN, q4.Q4_F32)
    check_plain(W, X, eids, Y, what="E=1 R=1")


def test_256_experts_mostly_empty():
    counts = [0] * 256
    for e, c in [(0, 2), (77, 1), (128, 19), (255, 4)]:
        counts[e] = c
    N, K = 128, 128
    W = q4synth.q4_matrix(350, N, K, experts=256)
    X = q4synth.activations(351, sum(counts), K)
    Y, eids = run_gemm(W, X, counts, N, K, q4.Q4_GEMV_PLAIN, q4.Q4_F16)
    check_plain(W, X, eids, Y, fp16_out=True, what="E=256")


@pytest.mark.parametrize("mode,K,counts", [(q4.Q4_GEMV_GLU, 8192, [3, 130]), (q4.Q4_GEMV_PLAIN, 9728, [3, 130]),
                                            (q4.Q4_GEMV_GLU, 1088, [3, 130]), (q4.Q4_GEMV_PLAIN, 1600, [3, 130]),
                                            (q4.Q4_GEMV_GLU, 6016, [2, 5, 0, 9]),
                                            (q4.Q4_GEMV_PLAIN, 8384, [2, 5, 0, 9])])
def test_large_k(mode, K, counts):
    """128-token units (A in shared memory) read their scales and biases from
    global memory once staging them would take more than 32 KB, so K is not
    bounded there (GLU at 8192, PLAIN at 9728; at 1088 and 1600 the group
    count is not a multiple of 4, which takes the one-group loads instead of
    the four-group ones); 32-token units stage them in shared memory, whose
    room bounds K (GLU up to about 6300, PLAIN about 8800 at 227 KB a block):
    a K just below that."""
    n_out = 128
    rows = 2 * n_out if mode == q4.Q4_GEMV_GLU else n_out
    W = q4synth.q4_matrix(360 + K, rows, K, experts=len(counts))
    X = q4synth.activations(361 + K, sum(counts), K)
    Y, eids = run_gemm(W, X, counts, n_out, K, mode, q4.Q4_F16)
    if mode == q4.Q4_GEMV_GLU:
        check_glu(W, X, eids, Y, n_out, what=f"GLU K={K}")
    else:
        check_plain(W, X, eids, Y, fp16_out=True, what=f"plain K={K}")


def test_few_tokens_per_expert_at_a_larger_k():
    """Few routed rows per expert take 32-token units (A in tensor memory,
    scales and biases staged) at K = 3584 in GLU mode."""
    n_out, K, counts = 128, 3584, [2, 5, 0, 9]
    W = q4synth.q4_matrix(370, 2 * n_out, K, experts=len(counts))
    X = q4synth.activations(371, sum(counts), K)
    Y, eids = run_gemm(W, X, counts, n_out, K, q4.Q4_GEMV_GLU, q4.Q4_F16)
    check_glu(W, X, eids, Y, n_out, what=f"GLU K={K}, 32-token units")


def test_k_beyond_shared_memory_is_refused():
    """32-token units (8 routed rows for one expert) at K = 6656 in GLU mode:
    the staged scales and biases leave no room for two input stages."""
    E, N, K, R = 1, 128, 6656, 8
    Wq = torch.zeros(E, 2 * N, K // 8, dtype=torch.int32, device="cuda")
    s = torch.zeros(E, 2 * N, K // 64, dtype=torch.float16, device="cuda")
    X = torch.zeros(R, K, dtype=torch.float16, device="cuda")
    ids = torch.zeros(R, dtype=torch.int32, device="cuda")
    off = torch.tensor([0, R], dtype=torch.int32, device="cuda")
    Y = torch.zeros(R, N, dtype=torch.float16, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.q4_moe_gemm(Wq, s, s, X, ids, off, Y, E, N, K, R, q4.Q4_GEMV_GLU, q4.Q4_F16)
    assert ei.value.name == "Q4_ERR_UNSUPPORTED"


def test_general_scales_and_biases():
    g = np.random.default_rng(320)
    E, N, K = 3, 128, 128
    counts = [5, 40, 9]
    Wq = g.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint32)
    s = (g.standard_normal((E, N, K // 64)) * 0.05).astype(np.float16)
    b = (g.standard_normal((E, N, K // 64)) * 0.2).astype(np.float16)
    W = q4synth.Q4Matrix(Wq, s, b)
    X = g.standard_normal((sum(counts), K)).astype(np.float16)
    Y, eids = run_gemm(W, X, counts, N, K, q4.Q4_GEMV_PLAIN, q4.Q4_F32)
    check_plain(W, X, eids, Y, what="general s,b")


def test_deterministic():
    N, K = 128, 256
    W = q4synth.q4_matrix(330, N, K, experts=len(COUNTS))
    X = q4synth.activations(331, sum(COUNTS), K)
    Y1, _ = run_gemm(W, X, COUNTS, N, K, q4.Q4_GEMV_PLAIN, q4.Q4_F32)
    Y2, _ = run_gemm(W, X, COUNTS, N, K, q4.Q4_GEMV_PLAIN, q4.Q4_F32)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))


def test_bad_expert_ids_latch_device_check():
    N, K = 128, 64
    counts = [4, 4]
    W = q4synth.q4_matrix(340, N, K, experts=2)
    X = q4synth.activations(341, 8, K)
    off = offsets_from_counts(counts)
    eids = np.array([0, 0, 0, 1, 1, 1, 1, 1], np.int32)   # row 3 belongs to expert 0
    Y = torch.empty(8, N, device="cuda")
    q4.q4_moe_gemm(*dev_q4(W), torch_dev(X), torch_dev(eids), torch_dev(off), Y, 2, N, K, 8, q4.Q4_GEMV_PLAIN,
                   q4.Q4_F32)
    assert q4.q4_device_status() == -7
    assert q4.q4_device_status() == 0      # cleared after reading


# ------------------------------------------------------------ full layer ---

SHAPE = q4synth.QWEN3_30B_A3B_MOE


@pytest.fixture(scope="module")
def moe():
    gu, dn = q4synth.moe_weights(SHAPE)
    return gu, dn, dev_q4(gu), dev_q4(dn)


def gpu_layer(moe, T, seed):
    gu, dn, dgu, ddn = moe
    E, k, H, F = SHAPE.experts, SHAPE.topk, SHAPE.hidden, SHAPE.ffn
    logits = q4synth.router_logits(seed, T, E)
    X = q4synth.activations(seed + 1, T, H)
    R = T * k
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    tok = torch.empty(R, dtype=torch.int32, device="cuda")
    eid = torch.empty(R, dtype=torch.int32, device="cuda")
    pos = torch.empty(T, k, dtype=torch.int32, device="cuda")
    nws = q4.q4_moe_route_workspace_bytes(T, E, k)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    q4.q4_moe_route(torch_dev(logits), T, E, k, ids, w, off, tok, eid, pos, ws, nws)
    Xs = torch.empty(R, H, dtype=torch.float16, device="cuda")
    q4.q4_moe_gather(torch_dev(X), T, H, tok, R, Xs)
    Hh = torch.full((R, F), float("nan"), dtype=torch.float16, device="cuda")
    q4.q4_moe_gemm(*dgu, Xs, eid, off, Hh, E, F, H, R, q4.Q4_GEMV_GLU, q4.Q4_F16)
    Y = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_moe_gemm(*ddn, Hh, eid, off, Y, E, H, F, R, q4.Q4_GEMV_PLAIN, q4.Q4_F32)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_moe_combine(Y, q4.Q4_F32, H, pos, w, T, k, out, q4.Q4_F32)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    c = lambda t: t.cpu().numpy()
    return dict(logits=logits, X=X, Xs=c(Xs), H=c(Hh.float()), Y=c(Y), out=c(out), eid=c(eid), tok=c(tok),
                pos=c(pos), w=c(w), off=c(off))


@pytest.mark.parametrize("T", [128, 512, 2048])
def test_qwen3_30b_a3b_layer_sampled_rows(moe, T):
    gu, dn = moe[0], moe[1]
    g = gpu_layer(moe, T, q4synth.BASE_SEED + 70 + T)
    r = oracle.moe_route(g["logits"], SHAPE.topk)
    assert np.array_equal(g["off"], r["offsets"]) and np.array_equal(g["tok"], r["token_of"])
    assert np.array_equal(g["Xs"].view(np.uint16), g["X"][g["tok"]].view(np.uint16))
    # the first and the last routed row of every expert that has rows (unit and
    # token-tile edges), and 96 more at random
    R = T * SHAPE.topk
    off = g["off"]
    nonempty = np.nonzero(off[1:] > off[:-1])[0]
    edges = np.concatenate([off[nonempty], off[nonempty + 1] - 1])
    rows = np.unique(np.concatenate([edges, np.random.default_rng(T).integers(0, R, 96)]))
    check_glu(gu, g["Xs"].astype(np.float16), g["eid"], g["H"], SHAPE.ffn, rows=rows, what=f"gate/up T={T}")
    check_plain(dn, g["H"].astype(np.float16), g["eid"], g["Y"], rows=rows, what=f"down T={T}")


def test_qwen3_30b_a3b_layer_end_to_end_small_T(moe):
    gu, dn = moe[0], moe[1]
    T = 24
    g = gpu_layer(moe, T, q4synth.BASE_SEED + 99)
    r = oracle.moe_route(g["logits"], SHAPE.topk)
    Xs = g["X"][r["token_of"]]
    _, _, _, _, act = oracle.moe_gate_up_rows(gu, Xs, r["expert_of"], SHAPE.ffn)
    Yr, _ = oracle.moe_down_rows(dn, oracle.fp16(act), r["expert_of"])
    out, mag = oracle.moe_combine(Yr, r["pos"], r["weights"])
    rel = np.linalg.norm(g["out"] - out) / np.linalg.norm(out)
    assert rel <= 1e-3, rel
