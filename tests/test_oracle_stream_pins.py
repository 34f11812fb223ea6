"""Pins for the oracle's decode-stream and MoE compositions: special cases that
reduce to elementwise arithmetic (diagonal weights), a hand-worked routing
fixture, an independent library sort, and invariants."""
import os

import numpy as np
import pytest

import oracle
import q4synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def diag_matrix(codes, scales):
    """Square W with w[n][n] = s_n * (c_n - 8) and exact zeros elsewhere
    (code 8 with bias -8 s gives w = 0).  One group per row (K = 64)."""
    n = len(codes)
    assert n == 64
    Wq = np.full((n, 8), 0x88888888, np.uint32)
    for i, c in enumerate(codes):
        w = i // 8
        sh = 4 * (i % 8)
        Wq[i, w] = (int(Wq[i, w]) & ~(0xF << sh) & 0xFFFFFFFF) | (c << sh)
    s = np.array(scales, np.float16).reshape(n, 1)
    b = (-8.0 * s.astype(np.float64)).astype(np.float16)
    return q4synth.Q4Matrix(Wq, s, b)


def diag_values(m):
    codes = [(int(m.Wq[i, i // 8]) >> (4 * (i % 8))) & 0xF for i in range(64)]
    return m.scales[:, 0].astype(np.float64) * (np.array(codes) - 8)


def test_diagonal_decode_step_reduces_to_elementwise():
    """With diagonal weights every GEMV is an elementwise product, so the whole
    stack (norms, residuals, SiLU*up, fp16 stores) can be written out directly."""
    g = np.random.default_rng(3)
    layers = []
    for _ in range(2):
        d = {}
        for nm in ("q", "k", "v", "o", "gate", "up", "down"):
            d[nm] = diag_matrix(list(g.integers(0, 16, 64)), list(np.exp2(g.integers(-4, 1, 64)) * 0.75))
        d["attn_norm"] = (g.random(64) + 0.5).astype(np.float16)
        d["ffn_norm"] = (g.random(64) + 0.5).astype(np.float16)
        layers.append(d)
    lm = diag_matrix(list(g.integers(0, 16, 64)), list(np.exp2(g.integers(-3, 0, 64))))
    fin = (g.random(64) + 0.5).astype(np.float16)
    x = q4synth.activations(9, 2, 64)
    eps = 1e-5
    logits, A, h_last = oracle.decode_step(layers, lm, x, final_norm=fin, eps=eps)

    f16 = lambda v: np.asarray(v, np.float64).astype(np.float16).astype(np.float64)
    nrm = lambda v, w: v / np.sqrt((v * v).mean(axis=1, keepdims=True) + eps) * w.astype(np.float64)
    h = x.astype(np.float64)
    for d in layers:
        q = f16(diag_values(d["q"]) * nrm(h, d["attn_norm"]))
        hm = f16(h + diag_values(d["o"]) * q)
        n2 = nrm(hm, d["ffn_norm"])
        gg = diag_values(d["gate"]) * n2
        act = f16(gg / (1 + np.exp(-gg)) * (diag_values(d["up"]) * n2))
        h = f16(hm + diag_values(d["down"]) * act)
    want = diag_values(lm) * nrm(h, fin)
    assert np.array_equal(h_last.astype(np.float64), h)
    assert np.allclose(logits, want, rtol=1e-15, atol=0)


def test_zero_o_and_down_leave_h_unchanged():
    shape = q4synth.tiny_decode_shape(n_layers=2, hidden=128, q=192, kv=64, ffn=256, vocab=80)
    layers, lm = q4synth.decode_weights(shape, base_seed=77)
    for d in layers:
        for nm in ("o", "down"):
            m = d[nm]
            m.Wq[:] = 0x88888888
            m.biases[:] = (-8.0 * m.scales.astype(np.float64)).astype(np.float16)
    x = q4synth.activations(78, 1, 128)
    logits, _, h = oracle.decode_step(layers, lm, x)
    direct, _ = oracle.gemv(lm.Wq, lm.scales, lm.biases, oracle.rmsnorm(x))
    assert np.array_equal(h, x) and np.array_equal(logits, direct)


def test_rmsnorm_closed_forms():
    eps = 1e-6
    for c in (0.5, -3.0, 1000.0):
        v = np.full((1, 256), c)
        r = oracle.rmsnorm(v, eps=eps)
        assert np.allclose(r, np.sign(c) / np.sqrt(1 + eps / c ** 2), rtol=1e-15, atol=0)
    h = q4synth.activations(5, 3, 512).astype(np.float64)
    r = oracle.rmsnorm(h, eps=0.0)
    assert np.allclose((r * r).mean(axis=1), 1.0, rtol=1e-14)          # unit mean square
    assert np.allclose(oracle.rmsnorm(8.0 * h, eps=0.0), r, rtol=1e-14)  # scale invariance
    w = np.linspace(0.5, 2, 512)
    assert np.allclose(oracle.rmsnorm(h, w, eps=0.0), r * w, rtol=1e-15)
    assert np.all(np.sign(r) == np.sign(h))


# ---------------------------------------------------------------- routing --

def load_routing_fixture():
    d = {"logits": {}, "ids": {}, "pos": {}}
    with open(os.path.join(GOLDEN, "moe_routing_worked_example.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] in ("E", "topk"):
                d[t[0]] = int(t[1])
            elif t[0] == "logits":
                d["logits"][int(t[1])] = [float(v) for v in t[2:]]
            elif t[0] in ("ids", "pos"):
                d[t[0]][int(t[1])] = [int(v) for v in t[2:]]
            else:
                d[t[0]] = [int(v) for v in t[1:]]
    T = len(d["logits"])
    d["logits"] = np.array([d["logits"][t] for t in range(T)], np.float16)
    d["ids"] = np.array([d["ids"][t] for t in range(T)])
    d["pos"] = np.array([d["pos"][t] for t in range(T)])
    return d


def test_routing_hand_worked_example():
    fx = load_routing_fixture()
    r = oracle.moe_route(fx["logits"], fx["topk"])
    assert np.array_equal(r["ids"], fx["ids"])
    assert np.array_equal(r["offsets"], fx["offsets"])
    assert np.array_equal(r["token_of"], fx["token_of"])
    assert np.array_equal(r["expert_of"], fx["expert_of"])
    assert np.array_equal(r["pos"], fx["pos"])
    assert np.allclose(r["weights"][0], 1 / 3, rtol=0, atol=1e-15)
    assert np.allclose(r["weights"][2], 1 / 3, rtol=0, atol=1e-15)
    z = 1 + np.exp(-1.0) + np.exp(-2.0)
    assert np.allclose(r["weights"][1], [1 / z, np.exp(-1.0) / z, np.exp(-2.0) / z], rtol=1e-15)


def test_routing_matches_library_sort():
    g = np.random.default_rng(21)
    T, E, k = 40, 16, 4
    logits = g.integers(-3, 4, size=(T, E)).astype(np.float16) * np.float16(0.5)  # many ties
    r = oracle.moe_route(logits, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        assert np.array_equal(r["ids"][t], order[:k])
    keys = np.lexsort((r["rank_of"], r["token_of"], r["expert_of"]))
    assert np.array_equal(keys, np.arange(T * k))        # rows already sorted by (e, t, k)


def test_routing_invariants_full_size():
    T, E, k = 128, 128, 8
    logits = q4synth.router_logits(31, T, E)
    r = oracle.moe_route(logits, k)
    R = T * k
    assert r["offsets"][0] == 0 and r["offsets"][-1] == R
    assert np.all(np.diff(r["offsets"]) >= 0)
    assert np.array_equal(np.diff(r["offsets"]), np.bincount(r["ids"].ravel(), minlength=E))
    for t in range(T):
        assert len(set(r["ids"][t])) == k
        vals = logits[t, r["ids"][t]].astype(np.float64)
        assert np.all(np.diff(vals) <= 0)
        assert vals[-1] >= np.sort(logits[t].astype(np.float64))[-k]
        assert abs(r["weights"][t].sum() - 1) < 1e-14 and np.all(np.diff(r["weights"][t]) <= 0)
        for kk in range(k):
            row = r["pos"][t, kk]
            assert r["token_of"][row] == t and r["rank_of"][row] == kk
            assert r["expert_of"][row] == r["ids"][t, kk]
    for e in range(E):
        assert np.all(r["expert_of"][r["offsets"][e]:r["offsets"][e + 1]] == e)


def test_combine_with_one_hot_rows():
    fx = load_routing_fixture()
    r = oracle.moe_route(fx["logits"], fx["topk"])
    R = r["token_of"].size
    Y = np.eye(R)
    out, _ = oracle.moe_combine(Y, r["pos"], r["weights"])
    for t in range(out.shape[0]):
        want = np.zeros(R)
        for kk in range(fx["topk"]):
            want[r["pos"][t, kk]] = r["weights"][t, kk]
        assert np.array_equal(out[t], want)


def test_expert_gate_up_split_matches_full_gemv():
    shape = q4synth.MoEShape("tiny-moe", 128, 4, 64, 2)
    gu, dn = q4synth.moe_weights(shape, base_seed=55)
    X = q4synth.activations(56, 3, 128)
    experts = np.array([2, 0, 3])
    g, Ag, u, Au, act = oracle.moe_gate_up_rows(gu, X, experts, 64)
    for i, e in enumerate(experts):
        full, _ = oracle.gemv(gu.Wq[e], gu.scales[e], gu.biases[e], X[i:i + 1])
        assert np.array_equal(g[i], full[0, :64]) and np.array_equal(u[i], full[0, 64:])
    H = oracle.fp16(act)
    y, _ = oracle.moe_down_rows(dn, H, experts)
    for i, e in enumerate(experts):
        full, _ = oracle.gemv(dn.Wq[e], dn.scales[e], dn.biases[e], H[i:i + 1])
        assert np.array_equal(y[i], full[0])


# ---------------------------------------------------------------- prefill --

def diag_stack(seed, n_layers=2):
    g = np.random.default_rng(seed)
    layers = []
    for _ in range(n_layers):
        d = {}
        for nm in ("q", "k", "v", "o", "gate", "up", "down"):
            d[nm] = diag_matrix(list(g.integers(0, 16, 64)), list(np.exp2(g.integers(-4, 1, 64)) * 0.75))
        d["attn_norm"] = (g.random(64) + 0.5).astype(np.float16)
        d["ffn_norm"] = (g.random(64) + 0.5).astype(np.float16)
        layers.append(d)
    lm = diag_matrix(list(g.integers(0, 16, 64)), list(np.exp2(g.integers(-3, 0, 64))))
    fin = (g.random(64) + 0.5).astype(np.float16)
    return layers, lm, fin


def test_diagonal_prefill_reduces_to_elementwise():
    """Diagonal weights again, now with both normalised activations stored in
    fp16 before their products, and the last token's logits."""
    layers, lm, fin = diag_stack(13)
    x = q4synth.activations(14, 5, 64)
    eps = 1e-5
    h_o, logits, A = oracle.prefill(layers, lm, x, final_norm=fin, eps=eps)

    f16 = lambda v: np.asarray(v, np.float64).astype(np.float16).astype(np.float64)
    nrm = lambda v, w: v / np.sqrt((v * v).mean(axis=1, keepdims=True) + eps) * w.astype(np.float64)
    h = x.astype(np.float64)
    for d in layers:
        n = f16(nrm(h, d["attn_norm"]))
        q = f16(diag_values(d["q"]) * n)
        hm = f16(h + diag_values(d["o"]) * q)
        n2 = f16(nrm(hm, d["ffn_norm"]))
        gg = diag_values(d["gate"]) * n2
        act = f16(gg / (1 + np.exp(-gg)) * (diag_values(d["up"]) * n2))
        h = f16(hm + diag_values(d["down"]) * act)
    assert np.array_equal(h_o.astype(np.float64), h)
    want = diag_values(lm) * nrm(h[-1:], fin)
    assert np.allclose(logits, want, rtol=1e-15, atol=0)


def test_prefill_tokens_are_independent():
    """No attention in this stack: each token's result is that of the token
    alone, and the logits are those of the last token."""
    shape = q4synth.tiny_decode_shape(n_layers=2, hidden=128, q=256, kv=128, ffn=256, vocab=96)
    layers, lm = q4synth.decode_weights(shape, base_seed=91)
    x = q4synth.activations(92, 4, 128)
    h_all, y_all, _ = oracle.prefill(layers, lm, x)
    for t in range(4):
        h_t, y_t, _ = oracle.prefill(layers, lm, x[t:t + 1])
        assert np.array_equal(h_all[t], h_t[0])
    assert np.array_equal(y_all, y_t)


def test_prefill_equals_decode_when_norms_are_fp16_exact():
    """With eps = 0, zero o and down products and a constant-magnitude x,
    rms(h) * gamma = sign(h) * gamma is exact in fp16, so storing the norm in
    fp16 changes nothing and the prefill stream equals the decode stream."""
    shape = q4synth.tiny_decode_shape(n_layers=2, hidden=128, q=128, kv=128, ffn=256, vocab=64)
    layers, lm = q4synth.decode_weights(shape, base_seed=93)
    for d in layers:
        for nm in ("o", "down"):
            m = d[nm]
            m.Wq[:] = 0x88888888
            m.biases[:] = (-8.0 * m.scales.astype(np.float64)).astype(np.float16)
        d["attn_norm"] = np.linspace(0.5, 1.5, 128).astype(np.float16)
        d["ffn_norm"] = np.linspace(1.5, 0.5, 128).astype(np.float16)
    g = np.random.default_rng(94)
    x = (np.where(g.random((3, 128)) < 0.5, -1.0, 1.0) * 0.75).astype(np.float16)
    h_p, y_p, _ = oracle.prefill(layers, lm, x, eps=0.0)
    y_d, _, h_d = oracle.decode_step(layers, lm, x, eps=0.0)
    assert np.array_equal(h_p, h_d)
    assert np.array_equal(y_p, y_d[-1:])
    for d in layers:   # and the stage values agree too
        a = oracle.prefill_layer(d, x, eps=0.0)
        b = oracle.decode_layer(d, x, eps=0.0)
        for nm in ("q", "k", "v", "h_mid", "act", "h"):
            assert np.array_equal(a[nm], b[nm]), nm
