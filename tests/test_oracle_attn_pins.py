"""Pins for the oracle's rotary embedding and decode attention: a hand-worked
rotation, identities of rotations (position 0, norms, composition), and
special cases of attention with closed forms (one position, equal keys, a
dominant key, the grouped-query head mapping, two keys whose scaled scores
ln 3 and 0 weigh the values exactly 3/4 and 1/4 -- which fixes the 1/sqrt(d)
score scale, with two planted scale mistakes that must fail it)."""
import math

import numpy as np
import pytest

import oracle


def test_rope_hand_worked_d4():
    """d = 4, theta = 10000: pair (0, 2) turns by pos, pair (1, 3) by pos/100."""
    x = np.array([1.0, 2.0, 3.0, 4.0])
    r = oracle.rope(x, 1, 4, theta=10000.0)
    c0, s0, c1, s1 = math.cos(1.0), math.sin(1.0), math.cos(0.01), math.sin(0.01)
    want = [1 * c0 - 3 * s0, 2 * c1 - 4 * s1, 3 * c0 + 1 * s0, 4 * c1 + 2 * s1]
    assert np.allclose(r, want, rtol=0, atol=1e-15)


def test_rope_identities():
    g = np.random.default_rng(1)
    d = 128
    x = g.standard_normal(4 * d)
    assert np.array_equal(oracle.rope(x, 0, d), x)                       # position 0
    for pos in (1, 17, 4095):
        r = oracle.rope(x, pos, d).reshape(4, d)
        xs = x.reshape(4, d)
        pn = lambda v: v[:, : d // 2] ** 2 + v[:, d // 2:] ** 2
        assert np.allclose(pn(r), pn(xs), rtol=1e-13)                    # each pair keeps its norm
    a, b = 37, 1000
    assert np.allclose(oracle.rope(oracle.rope(x, a, d), b, d), oracle.rope(x, a + b, d), rtol=0, atol=1e-11)
    # relative position: <rope(q, m), rope(k, n)> depends on m - n only
    q, k = g.standard_normal(d), g.standard_normal(d)
    d1 = oracle.rope(q, 50, d) @ oracle.rope(k, 20, d)
    d2 = oracle.rope(q, 130, d) @ oracle.rope(k, 100, d)
    assert abs(d1 - d2) < 1e-12


def caches(g, Hkv, n, d, max_seq=64):
    kc = np.zeros((Hkv, max_seq, d), np.float16)
    vc = np.zeros((Hkv, max_seq, d), np.float16)
    kc[:, :n] = g.standard_normal((Hkv, n, d)).astype(np.float16)
    vc[:, :n] = g.standard_normal((Hkv, n, d)).astype(np.float16)
    return kc, vc


def test_attention_single_position_returns_v():
    g = np.random.default_rng(2)
    d, Hq, Hkv = 64, 4, 2
    kc, vc = caches(g, Hkv, 1, d)
    q = g.standard_normal(Hq * d).astype(np.float16)
    a, A = oracle.attention(q, kc, vc, 1, d, pos=9)
    want = np.concatenate([vc[h // 2, 0] for h in range(Hq)]).astype(np.float64)
    assert np.array_equal(a, want) and np.array_equal(A, np.abs(want))


def test_attention_equal_keys_average_values():
    g = np.random.default_rng(3)
    d, Hq, Hkv, n = 64, 2, 1, 7
    kc, vc = caches(g, Hkv, n, d)
    kc[:, :n] = kc[:, :1]
    q = g.standard_normal(Hq * d).astype(np.float16)
    a, _ = oracle.attention(q, kc, vc, n, d, pos=3)
    want = vc[0, :n].astype(np.float64).mean(axis=0)
    assert np.allclose(a.reshape(Hq, d), want[None, :], rtol=0, atol=1e-14)


def test_attention_dominant_key_and_head_mapping():
    """Key j* of kv head 1 aligned with the rotated query of q heads 2 and 3
    at a large scale: their output is v_{j*} of kv head 1; q heads 0 and 1
    read kv head 0 (a different value) and are unaffected."""
    g = np.random.default_rng(4)
    d, Hq, Hkv, n, pos = 32, 4, 2, 9, 5
    kc, vc = caches(g, Hkv, n, d)
    q = g.standard_normal(Hq * d).astype(np.float16)
    qr = oracle.rope(q, pos, d).reshape(Hq, d)
    kc[1, 6] = (qr[2] * 64).astype(np.float16)   # q head 3 is not aligned: use head 2's query for both
    q = q.reshape(Hq, d).copy()
    q[3] = q[2]
    a, _ = oracle.attention(q.reshape(-1), kc, vc, n, d, pos)
    a = a.reshape(Hq, d)
    assert np.allclose(a[2], vc[1, 6], rtol=0, atol=1e-9) and np.allclose(a[3], vc[1, 6], rtol=0, atol=1e-9)
    ref0, _ = oracle.attention(q.reshape(-1)[: 2 * d], kc[:1], vc[:1], n, d, pos)
    assert np.array_equal(a[:2].reshape(-1), ref0)


def test_layer_with_attention_wiring():
    """Position 0: the cache takes k (rotation by 0 is the identity) and v,
    and attention over one position returns v.  Position 1: position 0 is
    kept, and a is a convex combination of the two values."""
    import q4synth
    shape = q4synth.tiny_decode_shape(n_layers=1, hidden=128, q=256, kv=128, ffn=256, vocab=64)
    layers, _ = q4synth.decode_weights(shape, base_seed=95)
    d, Hkv = 64, 2
    kc = np.zeros((Hkv, 8, d), np.float16)
    vc = np.zeros((Hkv, 8, d), np.float16)
    x0 = q4synth.activations(96, 1, 128)
    o0 = oracle.decode_layer_attn(layers[0], x0, kc, vc, 0, d)
    assert np.array_equal(kc[:, 0].reshape(-1), o0["k"]) and np.array_equal(vc[:, 0].reshape(-1), o0["v"])
    v_heads = o0["v"].reshape(Hkv, d)
    assert np.array_equal(o0["a"][0].reshape(4, d), v_heads[[0, 0, 1, 1]])
    k0 = kc[:, 0].copy()
    o1 = oracle.decode_layer_attn(layers[0], q4synth.activations(97, 1, 128), kc, vc, 1, d)
    assert np.array_equal(kc[:, 0], k0)
    assert np.array_equal(kc[:, 1].reshape(-1), oracle.fp16(oracle.rope(o1["k"], 1, d)))
    lo = np.minimum(vc[:, 0], vc[:, 1])[[0, 0, 1, 1]].reshape(-1)
    hi = np.maximum(vc[:, 0], vc[:, 1])[[0, 0, 1, 1]].reshape(-1)
    a = o1["a"][0].astype(np.float64)
    assert np.all(a >= lo - 1e-3 * np.abs(lo)) and np.all(a <= hi + 1e-3 * np.abs(hi))


def test_prefill_with_attention_equals_token_by_token_decode():
    """Prefill of T tokens with causal attention equals T decode steps with
    the normalised activations stored in fp16 -- checked against a decode
    composition built here from the pinned pieces (rmsnorm, gemv, rope,
    attention) one token at a time, with the caches filled in order."""
    import q4synth
    shape = q4synth.tiny_decode_shape(n_layers=2, hidden=128, q=256, kv=128, ffn=256, vocab=64)
    layers, lm = q4synth.decode_weights(shape, base_seed=97)
    d, Hkv, T, pos0 = 64, 2, 5, 3
    g = np.random.default_rng(98)
    base_k = g.standard_normal((2, Hkv, 16, d)).astype(np.float16)
    base_v = g.standard_normal((2, Hkv, 16, d)).astype(np.float16)
    caches_a = [(base_k[i].copy(), base_v[i].copy()) for i in range(2)]
    caches_b = [(base_k[i].copy(), base_v[i].copy()) for i in range(2)]
    x = q4synth.activations(99, T, 128)
    h_a, y_a, _ = oracle.prefill_attn(layers, lm, x, caches_a, pos0, d)
    hs = []
    for t in range(T):
        h = x[t:t + 1].astype(np.float16)
        for layer, (kc, vc) in zip(layers, caches_b):
            n = oracle.fp16(oracle.rmsnorm(h, layer.get("attn_norm")))
            qkv = {nm: oracle.fp16(oracle.gemv(layer[nm].Wq, layer[nm].scales, layer[nm].biases, n)[0])[0]
                   for nm in ("q", "k", "v")}
            kc[:, pos0 + t] = oracle.fp16(oracle.rope(qkv["k"], pos0 + t, d)).reshape(Hkv, d)
            vc[:, pos0 + t] = qkv["v"].reshape(Hkv, d)
            a = oracle.fp16(oracle.attention(qkv["q"], kc, vc, pos0 + t + 1, d, pos0 + t)[0])[None, :]
            hm = oracle.fp16(oracle.decode_o(layer, a, h)[0])
            n2 = oracle.fp16(oracle.rmsnorm(hm, layer.get("ffn_norm")))
            gg = oracle.gemv(layer["gate"].Wq, layer["gate"].scales, layer["gate"].biases, n2)[0]
            uu = oracle.gemv(layer["up"].Wq, layer["up"].scales, layer["up"].biases, n2)[0]
            act = oracle.fp16(oracle.silu(gg) * uu)
            h = oracle.fp16(oracle.decode_down(layer, act, hm)[0]).astype(np.float16)
        hs.append(h[0])
    assert np.array_equal(h_a, np.stack(hs))
    for (ka, va), (kb, vb) in zip(caches_a, caches_b):
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    # chunking: the first 2 tokens, then the other 3, from the same start
    caches_c = [(base_k[i].copy(), base_v[i].copy()) for i in range(2)]
    h1, _, _ = oracle.prefill_attn(layers, lm, x[:2], caches_c, pos0, d)
    h2, y2, _ = oracle.prefill_attn(layers, lm, x[2:], caches_c, pos0 + 2, d)
    assert np.array_equal(np.concatenate([h1, h2]), h_a) and np.array_equal(y2, y_a)


def _two_key_weights(d, mutant=0):
    """Two cached keys for one query head at position 0 (no rotation): the
    query is ln(3) on dimension 0, key 1 is sqrt(d) on dimension 0 and key 2
    is zero, so the scaled scores are ln 3 and 0 and the softmax weights are
    exactly 3/4 and 1/4.  Returns the output and the two values."""
    g = np.random.default_rng(5)
    kc = np.zeros((1, 4, d), np.float16)
    vc = np.zeros((1, 4, d), np.float16)
    kc[0, 0, 0] = math.sqrt(d)              # exact in fp16 for d = 16, 64, 256
    vc[0, :2] = g.standard_normal((2, d)).astype(np.float16)
    q = np.zeros(d)
    q[0] = math.log(3.0)
    a, _ = oracle.attention(q, kc, vc, 2, d, pos=0, mutant=mutant)
    return a, vc[0, 0].astype(np.float64), vc[0, 1].astype(np.float64)


def test_attention_score_scale_closed_form():
    """softmax(q.K^T / sqrt(d)): scores ln 3 and 0 weigh the values 3/4 and
    1/4, at three head sizes (so a fixed constant in place of sqrt(d) fails
    at least two of them)."""
    for d in (16, 64, 256):
        a, v1, v2 = _two_key_weights(d)
        assert np.allclose(a, 0.75 * v1 + 0.25 * v2, rtol=0, atol=1e-14), d


@pytest.mark.parametrize("mutant", [1, 2])
def test_attention_planted_scale_mistakes_are_caught(mutant):
    """Scores scaled by 1/d, or not scaled, fail the closed form."""
    a, v1, v2 = _two_key_weights(64, mutant=mutant)
    assert not np.allclose(a, 0.75 * v1 + 0.25 * v2, rtol=0, atol=1e-6)
