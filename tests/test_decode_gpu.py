"""GPU parity of q4_decode_step against the oracle's decode stream.

Per stage: each stage's output is compared with the oracle applied to the
GPU's own fp16 input of that stage (the tight per-element bound applies).
End to end: logits against the oracle's whole chain (relative L2 <= 1e-3).
Per-stage launches (CUDA-graph replay, direct launches, without programmatic
dependent launch, with the tagged hand-off) and the one persistent launch per
step give the same bits; pointer changes re-plan; tags stay correct past their
16-bit wrap."""
import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, dev_q4, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu


class _DevView:
    """A raw device pointer seen as an fp16 array (CUDA array interface)."""

    def __init__(self, ptr, shape):
        self.__cuda_array_interface__ = {"data": (int(ptr), False), "shape": tuple(shape), "typestr": "<f2",
                                         "version": 3, "strides": None}


def f16_from_ptr(ptr, M, n):
    torch.cuda.synchronize()
    return torch.as_tensor(_DevView(ptr, (M, n)), device="cuda").float().cpu().numpy()


class DevModel:
    """Weights on host (for the oracle) and device; norm weights random when
    ``gammas`` is set, else absent (ones)."""

    def __init__(self, shape, seed=q4synth.BASE_SEED, gammas=False, eps=0.0):
        self.shape = shape
        self.eps = eps
        self.layers, self.lm = q4synth.decode_weights(shape, seed)
        self.final_norm = None
        g = np.random.default_rng(seed + 5)
        if gammas:
            for d in self.layers:
                d["attn_norm"] = (g.random(shape.hidden) + 0.5).astype(np.float16)
                d["ffn_norm"] = (g.random(shape.hidden) + 0.5).astype(np.float16)
            self.final_norm = (g.random(shape.hidden) + 0.5).astype(np.float16)
        self.dl = []
        for d in self.layers:
            e = {k: (*dev_q4(v), v.N, v.K) for k, v in d.items() if not k.endswith("_norm")}
            for k in ("attn_norm", "ffn_norm"):
                if k in d:
                    e[k] = torch_dev(d[k])
            self.dl.append(e)
        self.dfin = None if self.final_norm is None else torch_dev(self.final_norm)
        self.dlm = (*dev_q4(self.lm), self.lm.N, self.lm.K)

    @property
    def oracle_eps(self):
        return self.eps if self.eps > 0 else oracle.DEFAULT_EPS

    def table(self, n_layers, M, flags=0, logits_dtype=q4.Q4_F32):
        t = q4.LayerTable(self.dl[:n_layers], self.dlm, hidden=self.shape.hidden, M=M, flags=flags,
                          logits_dtype=logits_dtype, final_norm=self.dfin, norm_eps=self.eps)
        n = q4.q4_decode_workspace_bytes(t)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        t.set_workspace(ws, n)
        return t

    def step(self, n_layers, x, flags=0, logits_dtype=q4.Q4_F32):
        M = x.shape[0]
        t = self.table(n_layers, M, flags, logits_dtype)
        logits = torch.full((M, self.shape.vocab), float("nan"),
                            dtype=torch.float32 if logits_dtype == q4.Q4_F32 else torch.float16, device="cuda")
        q4.q4_decode_step(t, torch_dev(x), logits)
        assert q4.q4_device_status() == 0
        b = q4.q4_decode_buffers(t)
        s = self.shape
        out = {"logits": logits.float().cpu().numpy(), "h": f16_from_ptr(b["h"], M, s.hidden)}
        if n_layers:
            out.update(h_mid=f16_from_ptr(b["h_mid"], M, s.hidden), q=f16_from_ptr(b["q"], M, s.q),
                       k=f16_from_ptr(b["k"], M, s.kv), v=f16_from_ptr(b["v"], M, s.kv),
                       act=f16_from_ptr(b["act"], M, s.ffn))
        t.release()
        return out


def check_layer(layer, h_in, out, rows=None, what="", eps=oracle.DEFAULT_EPS):
    """All four stages of one layer, each from the GPU's own stage input."""
    r = rows or {}
    qkv = oracle.decode_qkv(layer, h_in, rows=r.get("qkv"), eps=eps)
    for nm in ("q", "k", "v"):
        sel = r.get("qkv", {}).get(nm) if r.get("qkv") else None
        got = out[nm] if sel is None else out[nm][:, sel]
        assert_parity(got, *qkv[nm], fp16_out=True, what=f"{what} {nm}")
    hm_ref, A = oracle.decode_o(layer, out["q"], h_in, rows=r.get("hidden"))
    sel = r.get("hidden")
    assert_parity(out["h_mid"] if sel is None else out["h_mid"][:, sel], hm_ref, A, fp16_out=True,
                  what=f"{what} h_mid")
    g, Ag, u, Au, act_ref = oracle.decode_glu(layer, out["h_mid"], rows=r.get("ffn"), eps=eps)
    A = 1.1 * np.abs(u) * Ag + np.abs(oracle.silu(g)) * Au
    sel = r.get("ffn")
    assert_parity(out["act"] if sel is None else out["act"][:, sel], act_ref, A, fp16_out=True, what=f"{what} act")
    h_ref, A = oracle.decode_down(layer, out["act"], out["h_mid"], rows=r.get("hidden"))
    sel = r.get("hidden")
    assert_parity(out["h"] if sel is None else out["h"][:, sel], h_ref, A, fp16_out=True, what=f"{what} h")


@pytest.fixture(scope="module")
def tiny():
    return DevModel(q4synth.tiny_decode_shape(n_layers=3))


@pytest.fixture(scope="module")
def tiny_gamma():
    return DevModel(q4synth.tiny_decode_shape(n_layers=3, hidden=320, q=448, kv=64, ffn=832, vocab=517),
                    seed=q4synth.BASE_SEED + 50, gammas=True, eps=1e-5)


def run_every_stage(model, M, seed, flags=0):
    x = q4synth.activations(seed, M, model.shape.hidden)
    h_in = x
    eps = model.oracle_eps
    for n in range(1, model.shape.n_layers + 1):
        out = model.step(n, x, flags=flags)
        check_layer(model.layers[n - 1], h_in, out, what=f"layer {n - 1} M={M}", eps=eps)
        y_ref, A = oracle.decode_logits(model.lm, out["h"], model.final_norm, eps=eps)
        assert_parity(out["logits"], y_ref, A, what=f"logits after {n} layers")
        h_in = out["h"].astype(np.float16)
    l_ref, _, h_ref = oracle.decode_step(model.layers, model.lm, x, model.final_norm, eps=eps)
    rel = np.linalg.norm(out["logits"] - l_ref) / np.linalg.norm(l_ref)
    assert rel <= 1e-3, rel


@pytest.mark.parametrize("M", [1, 4])
def test_tiny_model_every_stage_and_end_to_end(tiny, M):
    run_every_stage(tiny, M, q4synth.BASE_SEED + 500 + M)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_norm_weights_every_stage_and_end_to_end(tiny_gamma, M):
    run_every_stage(tiny_gamma, M, q4synth.BASE_SEED + 600 + M)


PERSISTENT = q4.Q4_DECODE_PERSISTENT


@pytest.mark.parametrize("M", [1, 5])
def test_tagged_hand_off_every_stage_and_end_to_end(tiny_gamma, M):
    run_every_stage(tiny_gamma, M, q4synth.BASE_SEED + 650 + M, flags=q4.Q4_DECODE_TAGGED)


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8])
def test_persistent_step_every_stage_and_end_to_end(tiny_gamma, M):
    run_every_stage(tiny_gamma, M, q4synth.BASE_SEED + 660 + M, flags=PERSISTENT)


def test_zero_layers_is_lm_head(tiny):
    x = q4synth.activations(7, 2, tiny.shape.hidden)
    out = tiny.step(0, x)
    y_ref, A = oracle.decode_logits(tiny.lm, x)
    assert_parity(out["logits"], y_ref, A)


def test_fp16_logits(tiny):
    x = q4synth.activations(8, 1, tiny.shape.hidden)
    out = tiny.step(2, x, logits_dtype=q4.Q4_F16)
    y_ref, A = oracle.decode_logits(tiny.lm, out["h"])
    assert_parity(out["logits"], y_ref, A, fp16_out=True)


@pytest.mark.parametrize("M", [1, 4])
def test_persistent_and_per_stage_modes_agree(tiny, M):
    x = q4synth.activations(9, M, tiny.shape.hidden)
    a = tiny.step(3, x)
    for fl in (q4.Q4_DECODE_NO_GRAPH, q4.Q4_DECODE_NO_PDL, q4.Q4_DECODE_NO_PDL | q4.Q4_DECODE_NO_GRAPH,
               q4.Q4_DECODE_TAGGED, q4.Q4_DECODE_TAGGED | q4.Q4_DECODE_NO_GRAPH, PERSISTENT):
        o = tiny.step(3, x, flags=fl)
        for k in a:
            assert np.array_equal(a[k].view(np.uint32) if a[k].dtype == np.float32 else a[k],
                                  o[k].view(np.uint32) if o[k].dtype == np.float32 else o[k]), (fl, k)


@pytest.mark.parametrize("flags", [PERSISTENT, q4.Q4_DECODE_TAGGED])
def test_many_replays_stay_correct(tiny, flags):
    """Tags advance every step; 5200 steps of 13 stages (past the 16-bit tag
    space: 5200 * 13 > 65535) keep matching the oracle."""
    t = tiny.table(3, 1, flags=flags)
    xs = q4synth.activations(150, 1, tiny.shape.hidden)
    x_dev = torch_dev(xs)
    lg = torch.empty(1, tiny.shape.vocab, device="cuda")
    first = None
    for i in range(5200):
        q4.q4_decode_step(t, x_dev, lg)
        if i == 0:
            torch.cuda.synchronize()
            first = lg.cpu().numpy().copy()
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    last = lg.cpu().numpy()
    t.release()
    assert np.array_equal(first.view(np.uint32), last.view(np.uint32))
    ref, _, _ = oracle.decode_step(tiny.layers, tiny.lm, xs)
    assert np.linalg.norm(last - ref) / np.linalg.norm(ref) <= 1e-3


@pytest.mark.parametrize("flags", [0, PERSISTENT])
def test_replay_and_recapture(tiny, flags):
    M = 1
    t = tiny.table(3, M, flags=flags)
    xs = [q4synth.activations(100 + i, M, tiny.shape.hidden) for i in range(3)]
    l1 = torch.empty(M, tiny.shape.vocab, device="cuda")
    l2 = torch.empty(M, tiny.shape.vocab, device="cuda")
    x_dev = torch_dev(xs[0])
    outs = []
    for i, xv in enumerate(xs):
        x_dev.copy_(torch_dev(xv))            # same pointer: replay
        q4.q4_decode_step(t, x_dev, l1 if i < 2 else l2)   # new logits pointer: re-capture
        torch.cuda.synchronize()
        outs.append((l1 if i < 2 else l2).cpu().numpy().copy())
    t.release()
    for xv, o in zip(xs, outs):
        ref, _, _ = oracle.decode_step(tiny.layers, tiny.lm, xv)
        assert np.linalg.norm(o - ref) / np.linalg.norm(ref) <= 1e-3


@pytest.fixture(scope="module")
def qwen06():
    return DevModel(q4synth.QWEN3_0P6B)


def test_qwen3_0p6b_full_size(qwen06):
    """Full Qwen3-0.6B-shaped stream (28 layers + lm_head), M = 1: every stage
    of the last layer on sampled rows, sampled logits, and the end-to-end
    logits against the oracle's whole chain."""
    s = qwen06.shape
    x = q4synth.activations(q4synth.BASE_SEED + 777, 1, s.hidden)
    prev = qwen06.step(s.n_layers - 1, x)
    out = qwen06.step(s.n_layers, x)
    g = np.random.default_rng(3)
    rows = {"qkv": {"q": g.integers(0, s.q, 256), "k": g.integers(0, s.kv, 128), "v": g.integers(0, s.kv, 128)},
            "hidden": np.unique(g.integers(0, s.hidden, 256)), "ffn": np.unique(g.integers(0, s.ffn, 256))}
    check_layer(qwen06.layers[-1], prev["h"].astype(np.float16), out, rows=rows, what="last layer")
    lrows = np.unique(g.integers(0, s.vocab, 2048))
    y_ref, A = oracle.decode_logits(qwen06.lm, out["h"], rows=lrows)
    assert_parity(out["logits"][:, lrows], y_ref, A, what="logits sampled")
    l_ref, _, _ = oracle.decode_step(qwen06.layers, qwen06.lm, x)
    rel = np.linalg.norm(out["logits"] - l_ref) / np.linalg.norm(l_ref)
    assert rel <= 1e-3, rel
    persistent = qwen06.step(s.n_layers, x, flags=PERSISTENT)
    assert np.array_equal(out["logits"].view(np.uint32), persistent["logits"].view(np.uint32))


def full_size_check(model, M, seed, flags=0):
    """Every stage of the last layer on sampled rows (from the GPU's own input
    of that layer), sampled logits, and the end-to-end logits against the
    oracle's whole chain."""
    s = model.shape
    x = q4synth.activations(seed, M, s.hidden)
    prev = model.step(s.n_layers - 1, x, flags=flags)
    out = model.step(s.n_layers, x, flags=flags)
    g = np.random.default_rng(seed)
    rows = {"qkv": {"q": g.integers(0, s.q, 192), "k": g.integers(0, s.kv, 96), "v": g.integers(0, s.kv, 96)},
            "hidden": np.unique(g.integers(0, s.hidden, 192)), "ffn": np.unique(g.integers(0, s.ffn, 192))}
    check_layer(model.layers[-1], prev["h"].astype(np.float16), out, rows=rows, what=f"{s.name} last layer M={M}")
    lrows = np.unique(g.integers(0, s.vocab, 1024))
    y_ref, A = oracle.decode_logits(model.lm, out["h"], rows=lrows)
    assert_parity(out["logits"][:, lrows], y_ref, A, what=f"{s.name} logits sampled M={M}")
    l_ref, _, _ = oracle.decode_step(model.layers, model.lm, x)
    rel = np.linalg.norm(out["logits"] - l_ref) / np.linalg.norm(l_ref)
    assert rel <= 1e-3, (s.name, M, rel)


@pytest.fixture(scope="module")
def llama3b():
    return DevModel(q4synth.LLAMA32_3B)


@pytest.mark.parametrize("M", [1, 4])
def test_llama32_3b_full_size(llama3b, M):
    """The Llama-3.2-3B-shaped stream (28 layers, hidden 3072, lm_head 3072 ->
    128256) at M = 1 and in batched decode at M = 4."""
    full_size_check(llama3b, M, q4synth.BASE_SEED + 780 + M)


@pytest.fixture(scope="module")
def qwen4b():
    return DevModel(q4synth.QWEN3_4B)


def test_qwen3_4b_full_size(qwen4b):
    """The Qwen3-4B-shaped stream (36 layers, hidden 2560, lm_head 2560 -> 151936), M = 1."""
    full_size_check(qwen4b, 1, q4synth.BASE_SEED + 790)
