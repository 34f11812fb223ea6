"""GPU parity of decode attention (RoPE, KV-cache append, split attention,
merge) against the fp64 oracle, standalone and inside the decode step.

Standalone: positions on both sides of the 64-position chunk boundaries,
head groups of 1, 2 and 8 query heads per kv head, head_dim 64 and 128; the
appended cache position is checked to 1 ulp and every other position is
untouched; a position outside the cache latches a device-check status and
writes nothing.  In the step: several tokens from an empty cache and from a
prefilled 280-position context, per stage (the attention output against the
oracle fed the GPU's own q and caches) and end to end; graph replays advance
the device position and match uncaptured launches bit for bit."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, dev_q4, torch_dev, ulp16

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


def rand16(g, *shape):
    return g.standard_normal(shape).astype(np.float16)


def run_attention(q, k, v, kc, vc, pos, Hq, Hkv, d, theta=1e6):
    max_seq = kc.shape[1]
    dkc, dvc = torch_dev(kc), torch_dev(vc)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    a = torch.full((Hq * d,), float("nan"), dtype=torch.float16, device="cuda")
    nws = q4.q4_attention_workspace_bytes(Hq, d, max_seq)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    q4.q4_attention(torch_dev(q), torch_dev(k), torch_dev(v), dkc, dvc, dpos, Hq, Hkv, d, max_seq, a, ws, nws,
                    rope_theta=theta)
    st = q4.q4_device_status()
    return st, a.float().cpu().numpy(), dkc.cpu().numpy(), dvc.cpu().numpy(), int(dpos.item())


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 8, 128), (4, 4, 64), (16, 2, 128)])
@pytest.mark.parametrize("pos", [0, 1, 63, 64, 127, 128, 700])
def test_attention_standalone(Hq, Hkv, d, pos):
    g = np.random.default_rng(1000 + pos + Hq + d)
    max_seq = 768
    kc, vc = rand16(g, Hkv, max_seq, d), rand16(g, Hkv, max_seq, d)
    q, k, v = rand16(g, Hq * d), rand16(g, Hkv * d), rand16(g, Hkv * d)
    st, a, kc2, vc2, p2 = run_attention(q, k, v, kc, vc, pos, Hq, Hkv, d)
    assert st == 0 and p2 == pos
    want_k = oracle.fp16(oracle.rope(k, pos, d)).reshape(Hkv, d)
    assert np.all(np.abs(kc2[:, pos].astype(np.float64) - want_k) <= ulp16(want_k))
    assert np.array_equal(vc2[:, pos], v.reshape(Hkv, d))
    keep = np.ones(max_seq, bool)
    keep[pos] = False
    assert np.array_equal(kc2[:, keep], kc[:, keep]) and np.array_equal(vc2[:, keep], vc[:, keep])
    a_ref, A = oracle.attention(q, kc2, vc2, pos + 1, d, pos)
    assert_parity(a[None, :], a_ref[None, :], A[None, :], fp16_out=True, what=f"attention pos={pos}")


def test_attention_position_outside_cache():
    g = np.random.default_rng(1100)
    Hq, Hkv, d, max_seq = 4, 2, 64, 64
    kc, vc = rand16(g, Hkv, max_seq, d), rand16(g, Hkv, max_seq, d)
    for pos in (max_seq, -1):
        st, _, kc2, vc2, _ = run_attention(rand16(g, Hq * d), rand16(g, Hkv * d), rand16(g, Hkv * d), kc, vc, pos,
                                           Hq, Hkv, d)
        assert st == -7 and np.array_equal(kc2, kc) and np.array_equal(vc2, vc)


# ----------------------------------------------------- in the decode step ---

D_HEAD = 64


def attn_model(seed, n_layers=3):
    shape = q4synth.tiny_decode_shape(n_layers=n_layers, hidden=256, q=256, kv=128, ffn=512, vocab=1000)
    layers, lm = q4synth.decode_weights(shape, base_seed=seed)
    return shape, layers, lm


def gpu_attn_table(shape, layers, lm, max_seq, caches, pos, flags=0, hd=D_HEAD):
    dl, keep = [], []
    for d, (kc, vc) in zip(layers, caches):
        e = {k: (*dev_q4(d[k]), d[k].N, d[k].K) for k in ("q", "k", "v", "o", "gate", "up", "down")}
        e["k_cache"], e["v_cache"] = kc, vc
        dl.append(e)
    t = q4.LayerTable(dl, (*dev_q4(lm), lm.N, lm.K), hidden=shape.hidden, M=1,
                      flags=q4.Q4_DECODE_ATTENTION | flags, head_dim=hd, max_seq=max_seq, pos=pos)
    nws = q4.q4_decode_workspace_bytes(t)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    t.set_workspace(ws, nws)
    return t, ws


def read16(ws, ptr, n):
    off = ptr - ws.data_ptr()
    return ws[off:off + 2 * n].view(torch.float16).float().cpu().numpy()


def host_caches(shape, max_seq, fill, seed, d=D_HEAD):
    g = np.random.default_rng(seed)
    out = []
    for _ in range(shape.n_layers):
        kc = np.zeros((shape.kv // d, max_seq, d), np.float16)
        vc = np.zeros_like(kc)
        if fill:
            kc[:, :fill] = rand16(g, shape.kv // d, fill, d)
            vc[:, :fill] = rand16(g, shape.kv // d, fill, d)
        out.append((kc, vc))
    return out


@pytest.mark.parametrize("start", [0, 280])
def test_decode_step_with_attention(start):
    shape, layers, lm = attn_model(1200 + start)
    max_seq, steps = 320, 5
    hc = host_caches(shape, max_seq, start, 1201)
    dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
    pos = torch.tensor([start], dtype=torch.int32, device="cuda")
    t, ws = gpu_attn_table(shape, layers, lm, max_seq, dc, pos)
    logits = torch.empty(1, shape.vocab, device="cuda")
    for s in range(steps):
        x = q4synth.activations(1300 + s, 1, shape.hidden)
        q4.q4_decode_step(t, torch_dev(x), logits)
        assert q4.q4_device_status() == 0
        assert int(pos.item()) == start + s + 1
        # stage check: the last layer's attention output against the oracle fed
        # the GPU's own q and caches
        buf = q4.q4_decode_buffers(t)
        qg, ag = read16(ws, buf["q"], shape.q), read16(ws, buf["a"], shape.q)
        kl, vl = dc[-1][0].cpu().numpy(), dc[-1][1].cpu().numpy()
        a_ref, A_a = oracle.attention(qg.astype(np.float16), kl, vl, start + s + 1, D_HEAD, start + s)
        assert_parity(ag[None, :], a_ref[None, :], A_a[None, :], fp16_out=True, what=f"step {s} attention")
        y_ref, A, _ = oracle.decode_step_attn(layers, lm, x, hc, start + s, D_HEAD)
        r = np.linalg.norm(logits.cpu().numpy() - y_ref) / np.linalg.norm(y_ref)
        assert r <= 1e-3, (s, r)
    for (kc, vc), (dk, dv) in zip(hc, dc):
        got_k, got_v = dk.cpu().numpy().astype(np.float64), dv.cpu().numpy().astype(np.float64)
        sl = slice(start, start + steps)
        assert np.allclose(got_k[:, sl], kc[:, sl], rtol=2e-2, atol=2e-2)
        assert np.allclose(got_v[:, sl], vc[:, sl], rtol=2e-2, atol=2e-2)
        assert np.array_equal(got_k[:, :start], kc[:, :start].astype(np.float64))
    t.release()


def test_decode_attention_graph_replay_matches_direct_launches():
    shape, layers, lm = attn_model(1400, n_layers=2)
    max_seq = 300
    outs = []
    for flags in (0, q4.Q4_DECODE_NO_GRAPH):
        hc = host_caches(shape, max_seq, 260, 1401)
        dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
        pos = torch.tensor([260], dtype=torch.int32, device="cuda")
        t, _ = gpu_attn_table(shape, layers, lm, max_seq, dc, pos, flags)
        logits = torch.empty(1, shape.vocab, device="cuda")
        seq = []
        for s in range(4):
            q4.q4_decode_step(t, torch_dev(q4synth.activations(1500 + s, 1, shape.hidden)), logits)
            seq.append(logits.clone())
        assert q4.q4_device_status() == 0 and int(pos.item()) == 264
        outs.append((seq, [(k.clone(), v.clone()) for k, v in dc]))
        t.release()
    for a, b in zip(outs[0][0], outs[1][0]):
        assert torch.equal(a, b)
    for (ka, va), (kb, vb) in zip(outs[0][1], outs[1][1]):
        assert torch.equal(ka, kb) and torch.equal(va, vb)


# ---------------------------------------------------- prefill with attention ---

def prefill_attn_run(shape, layers, lm, dc, pos, x, chunk, d=D_HEAD):
    t, _ = gpu_attn_table(shape, layers, lm, dc[0][0].shape[1], dc, pos, hd=d)
    T = x.shape[0]
    h = torch_dev(x).clone()
    nws = q4.q4_prefill_workspace_bytes(t, chunk)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    lg = torch.full((shape.vocab,), float("nan"), device="cuda")
    q4.q4_prefill(t, h, T, chunk, lg, ws, nws)
    st = q4.q4_device_status()
    return t, st, h, lg, ws


@pytest.mark.parametrize("start,chunk", [(0, 16), (100, 16), (100, 64)])
def test_prefill_with_attention(start, chunk):
    shape, layers, lm = attn_model(1600 + start, n_layers=2)
    max_seq, T = 160, 37
    hc = host_caches(shape, max_seq, start, 1601)
    dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
    pos = torch.tensor([start], dtype=torch.int32, device="cuda")
    x = q4synth.activations(1602, T, shape.hidden)
    t, st, h, lg, ws = prefill_attn_run(shape, layers, lm, dc, pos, x, chunk)
    assert st == 0 and int(pos.item()) == start + T
    # stage check on the last layer's last chunk: each token's attention
    # output against the oracle fed the GPU's q and caches
    b = q4.q4_prefill_buffers(t, chunk, ws)
    C = T - (T - 1) // chunk * chunk
    t0 = T - C
    kl, vl = dc[-1][0].cpu().numpy(), dc[-1][1].cpu().numpy()
    for i in range(C):
        qg = read16(ws, b["q"] + 2 * i * shape.q, shape.q).astype(np.float16)
        ag = read16(ws, b["a"] + 2 * i * shape.q, shape.q)
        p = start + t0 + i
        a_ref, A_a = oracle.attention(qg, kl, vl, p + 1, D_HEAD, p)
        assert_parity(ag[None, :], a_ref[None, :], A_a[None, :], fp16_out=True, what=f"prefill attention t={t0 + i}")
    # end to end against the oracle's own prefill (its own caches)
    h_ref, y_ref, _ = oracle.prefill_attn(layers, lm, x, hc, start, D_HEAD)
    r_h = np.linalg.norm(h.float().cpu().numpy() - h_ref) / np.linalg.norm(h_ref.astype(np.float64))
    r_y = np.linalg.norm(lg.cpu().numpy() - y_ref[0]) / np.linalg.norm(y_ref[0])
    assert r_h <= 1e-3 and r_y <= 1e-3, (r_h, r_y)
    for (kc, vc), (dk, dv) in zip(hc, dc):
        gk, gv = dk.cpu().numpy().astype(np.float64), dv.cpu().numpy().astype(np.float64)
        sl = slice(start, start + T)
        assert np.allclose(gk[:, sl], kc[:, sl], rtol=2e-2, atol=2e-2)
        assert np.allclose(gv[:, sl], vc[:, sl], rtol=2e-2, atol=2e-2)
        assert np.array_equal(gk[:, :start], kc[:, :start].astype(np.float64))
        assert np.array_equal(gk[:, start + T:], kc[:, start + T:].astype(np.float64))
    t.release()


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_attention_several_query_blocks(d):
    # one chunk of 150 tokens (query blocks of 64, 64 and a ragged 22) after
    # 40 cached positions (key tiles of 64: 0..63, 64..127, 128..189); with
    # hidden 256, head_dim 128 gives 2 query heads on 1 kv head
    shape, layers, lm = attn_model(1900 + d, n_layers=2)
    max_seq, start, T, chunk = 200, 40, 150, 160
    hc = host_caches(shape, max_seq, start, 1901 + d, d)
    dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
    pos = torch.tensor([start], dtype=torch.int32, device="cuda")
    x = q4synth.activations(1902 + d, T, shape.hidden)
    t, st, h, lg, ws = prefill_attn_run(shape, layers, lm, dc, pos, x, chunk, d)
    assert st == 0 and int(pos.item()) == start + T
    b = q4.q4_prefill_buffers(t, chunk, ws)
    kl, vl = dc[-1][0].cpu().numpy(), dc[-1][1].cpu().numpy()
    for i in range(T):
        qg = read16(ws, b["q"] + 2 * i * shape.q, shape.q).astype(np.float16)
        ag = read16(ws, b["a"] + 2 * i * shape.q, shape.q)
        a_ref, A_a = oracle.attention(qg, kl, vl, start + i + 1, d, start + i)
        assert_parity(ag[None, :], a_ref[None, :], A_a[None, :], fp16_out=True, what=f"d={d} t={i}")
    h_ref, y_ref, _ = oracle.prefill_attn(layers, lm, x, hc, start, d)
    r_h = np.linalg.norm(h.float().cpu().numpy() - h_ref) / np.linalg.norm(h_ref.astype(np.float64))
    r_y = np.linalg.norm(lg.cpu().numpy() - y_ref[0]) / np.linalg.norm(y_ref[0])
    assert r_h <= 1e-3 and r_y <= 1e-3, (r_h, r_y)
    t.release()


@pytest.mark.parametrize("start,T,chunk,nan_tail", [(0, 300, 300, False), (77, 290, 160, True), (5, 37, 16, False)])
def test_prefill_attention_head_dim_128_tiles(start, T, chunk, nan_tail):
    """head_dim 128, 16 query heads on 8 kv heads: several 128-token query
    blocks and 128-position key tiles with ragged ends, a prompt split into
    chunks after cached positions; with nan_tail every cache row past the
    prompt holds NaN (stale rows must not reach the output)."""
    d = 128
    shape = q4synth.tiny_decode_shape(n_layers=1, hidden=256, q=16 * d, kv=8 * d, ffn=512, vocab=1000)
    layers, lm = q4synth.decode_weights(shape, base_seed=2100 + start)
    max_seq = start + T + 40
    hc = host_caches(shape, max_seq, start, 2101 + start, d)
    if nan_tail:
        for kc, vc in hc:
            kc[:, start + T:] = np.nan
            vc[:, start + T:] = np.nan
    dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
    pos = torch.tensor([start], dtype=torch.int32, device="cuda")
    x = q4synth.activations(2102 + start, T, shape.hidden)
    t, st, h, lg, ws = prefill_attn_run(shape, layers, lm, dc, pos, x, chunk, d)
    assert st == 0 and int(pos.item()) == start + T
    b = q4.q4_prefill_buffers(t, chunk, ws)
    C = T - (T - 1) // chunk * chunk
    t0 = T - C
    kl, vl = dc[-1][0].cpu().numpy(), dc[-1][1].cpu().numpy()
    for i in range(C):
        qg = read16(ws, b["q"] + 2 * i * shape.q, shape.q).astype(np.float16)
        ag = read16(ws, b["a"] + 2 * i * shape.q, shape.q)
        p = start + t0 + i
        a_ref, A_a = oracle.attention(qg, kl, vl, p + 1, d, p)
        assert_parity(ag[None, :], a_ref[None, :], A_a[None, :], fp16_out=True, what=f"t={t0 + i}")
    h_ref, y_ref, _ = oracle.prefill_attn(layers, lm, x, hc, start, d)
    r_h = np.linalg.norm(h.float().cpu().numpy() - h_ref) / np.linalg.norm(h_ref.astype(np.float64))
    r_y = np.linalg.norm(lg.cpu().numpy() - y_ref[0]) / np.linalg.norm(y_ref[0])
    assert r_h <= 1e-3 and r_y <= 1e-3, (r_h, r_y)
    t.release()


def test_prefill_then_decode_continues_the_sequence():
    shape, layers, lm = attn_model(1700, n_layers=2)
    max_seq, T = 96, 20
    hc = host_caches(shape, max_seq, 0, 1701)
    dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
    pos = torch.tensor([0], dtype=torch.int32, device="cuda")
    x = q4synth.activations(1702, T, shape.hidden)
    t, st, h, lg, _ = prefill_attn_run(shape, layers, lm, dc, pos, x, 8)
    assert st == 0 and int(pos.item()) == T
    oracle.prefill_attn(layers, lm, x, hc, 0, D_HEAD)
    logits = torch.empty(1, shape.vocab, device="cuda")
    for s in range(3):
        xs = q4synth.activations(1703 + s, 1, shape.hidden)
        q4.q4_decode_step(t, torch_dev(xs), logits)
        assert q4.q4_device_status() == 0 and int(pos.item()) == T + s + 1
        y_ref, _, _ = oracle.decode_step_attn(layers, lm, xs, hc, T + s, D_HEAD)
        r = np.linalg.norm(logits.cpu().numpy() - y_ref) / np.linalg.norm(y_ref)
        assert r <= 1e-3, (s, r)
    t.release()


def test_prefill_past_the_cache_is_refused_on_the_device():
    shape, layers, lm = attn_model(1800, n_layers=1)
    hc = host_caches(shape, 40, 0, 1801)
    dc = [(torch_dev(kc), torch_dev(vc)) for kc, vc in hc]
    pos = torch.tensor([35], dtype=torch.int32, device="cuda")  # 35 + 8 > 40: every chunk refused
    t, st, _, _, _ = prefill_attn_run(shape, layers, lm, dc, pos, q4synth.activations(1802, 16, shape.hidden), 8)
    assert st == -7
    for (kc, _), (dk, _) in zip(hc, dc):
        assert np.array_equal(dk.cpu().numpy(), kc)
    t.release()
