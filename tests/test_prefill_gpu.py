"""GPU parity of the dense prefill GEMM (q4_gemm: the tcgen05 grouped-GEMM
kernel with one expert, no routing) and of the chunked prefill of a layer
stack (q4_prefill) against the fp64 oracle.

The GEMM is compared on every element for ragged token counts (1 .. 300, so
one to three 128-token tiles with a ragged tail), both output types, GLU with
separate gate and up matrices, and the residual epilogue (also in place).  The
prefill is compared stage by stage on one layer (each stage fed the GPU's own
fp16 input), end to end on a small stack with a ragged last chunk, across
chunk sizes, and on sampled tokens of the Qwen3-0.6B-shaped stack."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, dev_q4, torch_dev, ulp16

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


def lin(m):
    return (*dev_q4(m), m.N, m.K)


def run_gemm(w, X, mode=q4.Q4_GEMV_PLAIN, out_dtype=q4.Q4_F32, up=None, residual=None, in_place=False,
             split=False):
    M, N = X.shape[0], w.N
    dt = torch.float16 if out_dtype == q4.Q4_F16 else torch.float32
    if in_place:
        Y = torch_dev(residual)
        res = Y
    else:
        Y = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        res = None if residual is None else torch_dev(residual)
    ws, nws = None, 0
    if split:
        nws = q4.q4_gemm_workspace_bytes(M, N, w.K, mode)
        assert nws > 0, "this shape should split K"
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    q4.q4_gemm(lin(w), torch_dev(X), Y, M, mode, out_dtype, up=None if up is None else lin(up), residual=res,
               workspace=ws, workspace_bytes=nws)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return Y.float().cpu().numpy()


def glu_ref(gate, up, X):
    g, Ag = oracle.gemv(gate.Wq, gate.scales, gate.biases, X)
    u, Au = oracle.gemv(up.Wq, up.scales, up.biases, X)
    return oracle.silu(g) * u, 1.1 * np.abs(u) * Ag + np.abs(oracle.silu(g)) * Au


# ------------------------------------------------------------------ GEMM ---

@pytest.mark.parametrize("M", [1, 17, 128, 200, 300])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_gemm_plain_every_element(M, out_dtype):
    N, K = 256, 320
    W = q4synth.q4_matrix(500 + M, N, K)
    X = q4synth.activations(501 + M, M, K)
    Y = run_gemm(W, X, out_dtype=out_dtype)
    y_ref, A = oracle.gemv(W.Wq, W.scales, W.biases, X)
    assert_parity(Y, y_ref, A, fp16_out=bool(out_dtype), what=f"gemm M={M}")


@pytest.mark.parametrize("M,K", [(300, 1600), (130, 4160)])
def test_gemm_scales_from_global_every_element(M, K):
    """K large enough that the dense GEMM reads each row's scales and biases
    from global memory instead of staging them: K = 1600 (25 groups: one-group
    loads) and 4160 (65 groups), plain with a residual in place and GLU, every
    element against the oracle."""
    N = 256
    W = q4synth.q4_matrix(580 + K, N, K)
    X = q4synth.activations(581 + K, M, K)
    y_ref, A = oracle.gemv(W.Wq, W.scales, W.biases, X)
    R = q4synth.activations(582 + K, M, N)
    Y = run_gemm(W, X, out_dtype=q4.Q4_F16, residual=R, in_place=True)
    r = R.astype(np.float64)
    assert_parity(Y, r + y_ref, A + np.abs(r), fp16_out=True, what=f"global scales M={M} K={K}")
    gate, up = q4synth.q4_matrix(583 + K, N, K), q4synth.q4_matrix(584 + K, N, K)
    H = run_gemm(gate, X, q4.Q4_GEMV_GLU, q4.Q4_F16, up=up)
    act, A2 = glu_ref(gate, up, X)
    assert_parity(H, act, A2, fp16_out=True, what=f"global scales glu M={M} K={K}")


@pytest.mark.parametrize("M", [5, 130])
def test_gemm_glu_separate_matrices(M):
    N, K = 384, 256
    gate, up = q4synth.q4_matrix(510, N, K), q4synth.q4_matrix(511, N, K)
    X = q4synth.activations(512, M, K)
    H = run_gemm(gate, X, q4.Q4_GEMV_GLU, q4.Q4_F16, up=up)
    act, A = glu_ref(gate, up, X)
    assert_parity(H, act, A, fp16_out=True, what=f"glu M={M}")


@pytest.mark.parametrize("in_place", [False, True])
def test_gemm_residual_epilogue(in_place):
    M, N, K = 150, 256, 512
    W = q4synth.q4_matrix(520, N, K)
    X = q4synth.activations(521, M, K)
    R = q4synth.activations(522, M, N)
    Y = run_gemm(W, X, out_dtype=q4.Q4_F16, residual=R, in_place=in_place)
    y, A = oracle.gemv(W.Wq, W.scales, W.biases, X)
    r = R.astype(np.float64)
    assert_parity(Y, r + y, A + np.abs(r), fp16_out=True, what=f"residual in_place={in_place}")


@pytest.mark.parametrize("M", [1, 130, 512])
def test_gemm_split_k_every_element(M):
    """Few output tiles: K split over units, fp32 partials, reduce kernel
    (plain fp32 and fp16, GLU, residual in place)."""
    N, K = 256, 2048
    W = q4synth.q4_matrix(550 + M, N, K)
    X = q4synth.activations(551 + M, M, K)
    y_ref, A = oracle.gemv(W.Wq, W.scales, W.biases, X)
    for out_dtype in (0, 1):
        Y = run_gemm(W, X, out_dtype=out_dtype, split=True)
        assert_parity(Y, y_ref, A, fp16_out=bool(out_dtype), what=f"split M={M}")
    R = q4synth.activations(552 + M, M, N)
    Y = run_gemm(W, X, out_dtype=q4.Q4_F16, residual=R, in_place=True, split=True)
    r = R.astype(np.float64)
    assert_parity(Y, r + y_ref, A + np.abs(r), fp16_out=True, what=f"split residual M={M}")
    gate, up = q4synth.q4_matrix(553, N, K), q4synth.q4_matrix(554, N, K)
    H = run_gemm(gate, X, q4.Q4_GEMV_GLU, q4.Q4_F16, up=up, split=True)
    act, A2 = glu_ref(gate, up, X)
    assert_parity(H, act, A2, fp16_out=True, what=f"split glu M={M}")


def test_gemm_qwen3_shapes_sampled_rows():
    """gate/up (GLU, K=1024 -> 3072) and down (K=3072 -> 1024) at 512 tokens,
    checked on sampled tokens."""
    M = 512
    gate, up = q4synth.q4_matrix(530, 3072, 1024), q4synth.q4_matrix(531, 3072, 1024)
    down = q4synth.q4_matrix(532, 1024, 3072)
    X = q4synth.activations(533, M, 1024)
    H = run_gemm(gate, X, q4.Q4_GEMV_GLU, q4.Q4_F16, up=up)
    rows = np.array([0, 1, 127, 128, 311, 511])
    act, A = glu_ref(gate, up, X[rows])
    assert_parity(H[rows], act, A, fp16_out=True, what="qwen gate/up")
    Hh = H.astype(np.float16)
    Y = run_gemm(down, Hh)
    y, A = oracle.gemv(down.Wq, down.scales, down.biases, Hh[rows])
    assert_parity(Y[rows], y, A, what="qwen down")


def test_gemm_zero_tokens_is_a_no_op():
    W = q4synth.q4_matrix(540, 128, 64)
    Y = torch.zeros(1, 128, device="cuda")
    q4.q4_gemm(lin(W), torch.zeros(1, 64, dtype=torch.float16, device="cuda"), Y, 0)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0 and float(Y.abs().sum()) == 0.0


def test_gemm_refusals():
    W = q4synth.q4_matrix(541, 200, 64)
    X = torch.zeros(4, 64, dtype=torch.float16, device="cuda")
    Y = torch.zeros(4, 256, dtype=torch.float16, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.q4_gemm(lin(W), X, Y, 4)                                  # N % 128
    assert ei.value.name == "Q4_ERR_UNSUPPORTED"
    W = q4synth.q4_matrix(542, 128, 64)
    U = q4synth.q4_matrix(543, 256, 64)
    for kw in (dict(mode=q4.Q4_GEMV_GLU, out_dtype=q4.Q4_F32, up=lin(W)),      # GLU writes fp16
               dict(mode=q4.Q4_GEMV_GLU, out_dtype=q4.Q4_F16, up=lin(U)),      # gate/up widths differ
               dict(mode=q4.Q4_GEMV_GLU, out_dtype=q4.Q4_F16),                 # no up matrix
               dict(out_dtype=q4.Q4_F32, residual=Y)):                         # residual needs fp16 out
        with pytest.raises(q4.Q4Error) as ei:
            q4.q4_gemm(lin(W), X, Y, 4, **kw)
        assert ei.value.name == "Q4_ERR_INVALID_ARG", kw


# --------------------------------------------------------------- prefill ---

def stack(shape, seed, norms=True):
    layers, lm = q4synth.decode_weights(shape, base_seed=seed)
    g = np.random.default_rng(seed + 1)
    if norms:
        for d in layers:
            d["attn_norm"] = (g.random(shape.hidden) + 0.5).astype(np.float16)
            d["ffn_norm"] = (g.random(shape.hidden) + 0.5).astype(np.float16)
    fin = (g.random(shape.hidden) + 0.5).astype(np.float16) if norms else None
    return layers, lm, fin


def gpu_table(layers, lm, fin, hidden):
    dl = []
    for d in layers:
        e = {k: lin(d[k]) for k in ("q", "k", "v", "o", "gate", "up", "down")}
        for k in ("attn_norm", "ffn_norm"):
            if d.get(k) is not None:
                e[k] = torch_dev(d[k])
        dl.append(e)
    return q4.LayerTable(dl, lin(lm), hidden=hidden, M=1, final_norm=None if fin is None else torch_dev(fin))


def run_prefill(table, x, chunk, logits=True):
    T, H = x.shape
    h = torch_dev(x).clone()
    nws = q4.q4_prefill_workspace_bytes(table, chunk)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    lg = torch.full((table.t.lm_head.N,), float("nan"), device="cuda") if logits else None
    q4.q4_prefill(table, h, T, chunk, lg, ws, nws)
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return h, lg, ws


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_prefill_one_layer_stage_by_stage():
    """Each stage against the oracle fed the GPU's own fp16 input (the
    workspace keeps the last chunk's n', q, k, v and act)."""
    shape = q4synth.tiny_decode_shape(n_layers=1, hidden=256, q=384, kv=128, ffn=640, vocab=1000)
    layers, lm, fin = stack(shape, 600)
    T = 40
    x = q4synth.activations(601, T, shape.hidden)
    table = gpu_table(layers, lm, fin, shape.hidden)
    h, lg, ws = run_prefill(table, x, chunk=T)
    d = layers[0]
    H, qN, kvN, F = shape.hidden, shape.q, shape.kv, shape.ffn
    off, sl = 0, {}
    for nm, w in (("n2", H), ("q", qN), ("k", kvN), ("v", kvN), ("act", F)):
        sl[nm] = ws[off:off + T * w * 2].view(torch.float16).view(T, w).float().cpu().numpy()
        off = (off + T * w * 2 + 255) // 256 * 256
    n_ref = oracle.fp16(oracle.rmsnorm(x, d["attn_norm"]))
    for nm in ("q", "k", "v"):
        y, A = oracle.gemv(d[nm].Wq, d[nm].scales, d[nm].biases, n_ref)
        assert_parity(sl[nm], y, A, fp16_out=True, what=f"stage {nm}")
    q_gpu = sl["q"].astype(np.float16)
    hm, A_hm = oracle.decode_o(d, q_gpu, x)
    hm16 = oracle.fp16(hm)
    n2_ref = oracle.fp16(oracle.rmsnorm(hm16, d["ffn_norm"]))
    # The GPU's own h' (overwritten in place) is within the product bound of
    # hm; n' inherits that error scaled by gamma / rms, plus its own rounding.
    rms = np.sqrt(np.mean(hm16.astype(np.float64) ** 2, axis=1, keepdims=True))
    gam = np.abs(d["ffn_norm"].astype(np.float64))[None, :]
    bound = (1e-3 * A_hm + ulp16(hm16)) * gam / rms * 1.01 + 2 * ulp16(n2_ref)
    assert np.all(np.abs(sl["n2"] - n2_ref) <= bound), "stage rmsnorm"
    n2 = sl["n2"].astype(np.float16)
    act, A = glu_ref(d["gate"], d["up"], n2)
    assert_parity(sl["act"], act, A, fp16_out=True, what="stage gate/up")
    hout, A = oracle.decode_down(d, sl["act"].astype(np.float16), hm16)
    assert_parity(h.float().cpu().numpy(), hout, A, fp16_out=True, what="stage down + residual")
    y, A = oracle.decode_logits(lm, h[-1:].cpu().numpy(), fin)
    assert_parity(lg.cpu().numpy()[None, :], y, A, what="last-token logits")


@pytest.mark.parametrize("chunk", [16, 37, 64])
def test_prefill_small_stack_end_to_end(chunk):
    shape = q4synth.tiny_decode_shape(n_layers=3, hidden=256, q=384, kv=128, ffn=640, vocab=1000)
    layers, lm, fin = stack(shape, 610)
    T = 37
    x = q4synth.activations(611, T, shape.hidden)
    h, lg, _ = run_prefill(gpu_table(layers, lm, fin, shape.hidden), x, chunk)
    h_ref, y_ref, _ = oracle.prefill(layers, lm, x, final_norm=fin)
    assert rel(h.float().cpu().numpy(), h_ref) <= 1e-3
    assert rel(lg.cpu().numpy(), y_ref[0]) <= 1e-3


def test_prefill_chunk_size_does_not_change_results():
    shape = q4synth.tiny_decode_shape(n_layers=2, hidden=256, q=384, kv=128, ffn=640, vocab=1000)
    layers, lm, fin = stack(shape, 620)
    x = q4synth.activations(621, 150, shape.hidden)
    table = gpu_table(layers, lm, fin, shape.hidden)
    outs = [run_prefill(table, x, c)[:2] for c in (16, 150, 1000)]
    for h, lg in outs[1:]:
        assert torch.equal(h, outs[0][0]) and torch.equal(lg, outs[0][1])


def test_prefill_qwen3_0p6b_sampled_tokens():
    """The Qwen3-0.6B-shaped stack (28 layers), 300 tokens in chunks of 128;
    the oracle runs the sampled tokens alone (tokens do not interact)."""
    shape = q4synth.QWEN3_0P6B
    layers, lm, fin = stack(shape, q4synth.BASE_SEED, norms=False)
    T = 300
    x = q4synth.activations(631, T, shape.hidden)
    h, lg, _ = run_prefill(gpu_table(layers, lm, fin, shape.hidden), x, chunk=128)
    hg = h.float().cpu().numpy()
    for t in (0, 127, 128, 299):
        h_ref, y_ref, _ = oracle.prefill(layers, lm, x[t:t + 1])
        assert rel(hg[t], h_ref[0]) <= 1e-3, t
        if t == T - 1:
            assert rel(lg.cpu().numpy(), y_ref[0]) <= 1e-3


def test_prefill_zero_tokens_and_refusals():
    shape = q4synth.tiny_decode_shape(n_layers=1, hidden=256, q=384, kv=128, ffn=640, vocab=1000)
    layers, lm, fin = stack(shape, 640)
    table = gpu_table(layers, lm, fin, shape.hidden)
    h, _, _ = run_prefill(table, np.zeros((0, shape.hidden), np.float16), 8, logits=False)
    nws = q4.q4_prefill_workspace_bytes(table, 8)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    hh = torch.zeros(4, shape.hidden, dtype=torch.float16, device="cuda")
    for args, name in (((hh, 4, 0, None, ws, nws), "Q4_ERR_INVALID_ARG"),       # chunk 0
                       ((hh, 4, 16, None, ws, nws), "Q4_ERR_INVALID_ARG"),      # workspace for chunk 8 only
                       ((hh, -1, 8, None, ws, nws), "Q4_ERR_INVALID_ARG")):
        with pytest.raises(q4.Q4Error) as ei:
            q4.q4_prefill(table, *args)
        assert ei.value.name == name, args
    bad = q4synth.tiny_decode_shape(n_layers=1, hidden=256, q=320, kv=128, ffn=640, vocab=1000)
    layers, lm, fin = stack(bad, 641)
    table = gpu_table(layers, lm, fin, bad.hidden)
    with pytest.raises(q4.Q4Error) as ei:
        q4.q4_prefill(table, hh, 4, 8, None, ws, nws)
    assert ei.value.name == "Q4_ERR_UNSUPPORTED"
