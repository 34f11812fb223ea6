"""Plain, slow CPU oracle for the Q4 decode matmul, its decode stream and the
MoE prefill layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It shares no
code with the CUDA library (``bit_quantized_gemv_q4_gb300``) and never imports
it; inputs come from ``q4synth`` (random draws only).

Pieces and the passages they follow:

* ``gemv``: the C oracle in ``q4_oracle.c`` -- the plain definition of the
  fused-dequant matmul (BaseRT: optimal LLM inference on Apple Silicon with
  native Metal, §3.3 "Kernel fusion and specialisation"), fp64, k in order.
* ``decode_*``: one decode step as a chain of GEMVs (BaseRT §3.3: GEMV for
  decode, M=1, fused QKV / FFN launches; MetalRT: AI inference performance
  optimisation on Apple Silicon, §2.2 decode throughput; "Mac on-device AI
  performance breakthrough", §2.2: the QKV products merged into one).  The pages
  do not give the dataflow between the GEMVs.  This oracle takes the plainest
  reading that keeps every matrix of the layer on the path and the values
  bounded, with the pre-norm RMSNorm of Qwen3/Llama-style layers (BaseRT §3.3
  lists normalisation among its kernels and fuses operator sequences of the
  attention path and FFN; MetalRT §5.1 keeps LayerNorm in fp32).  Without the
  norms the synthetic chain overflows fp16 within a few layers (SiLU*up grows
  quadratically):
      n     = rmsnorm(h) * g_attn   (fp64, not rounded: the GPU fuses it into
                                     the GEMV prologue and keeps it in fp32)
      q,k,v = Wq n, Wk n, Wv n      (stored fp16; k, v not consumed)
      a     = q                     (stand-in for attention, which is not on
                                     the matmul path)
      h'    = fp16(h + Wo a)
      act   = fp16(SiLU(Wg n') * (Wu n')),  n' = rmsnorm(h') * g_ffn
      h''   = fp16(h' + Wd act)
    and after the last layer  logits = Wlm (rmsnorm(h) * g_final).
    rmsnorm(v) = v / sqrt(mean(v^2) + eps); the norm weights g default to 1
    (their random-init value).
  Every activation the GPU stores as fp16 is rounded here too, RNE, from the
  fp64 value.
* ``moe_*``: routed-expert prefill (BaseRT abstract and Fig. 1: MoE prefill on
  a Qwen3-30B-A3B-shaped model; §3.4 "Prefill": GEMM for M>1).  The pages do not
  describe routing.  Reading taken: top-k of the fp16 router logits, ties to
  the lower expert index; weights = softmax over the k chosen logits; rows
  sorted stably by (expert, token, rank); per row gate/up -> fp16(SiLU(g)*u)
  -> down; output[t] = sum over ranks k = 0..topk-1 of p[t,k] * Y[pos[t,k]].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")


def lib_path(mutant: int = 0) -> str:
    """Path of the compiled C oracle (or of a planted-mistake build). Infrastructure:
    no passage."""
    return os.path.join(_HERE, "libq4oracle.so" if mutant == 0 else f"libq4oracle_mut{mutant}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP).  ``mutant`` > 0 builds a
    deliberately wrong variant used only by the pin tests."""
    out = lib_path(mutant)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", f"-DQ4O_MUTANT={mutant}",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_libs: dict[int, ctypes.CDLL] = {}


def _lib(mutant: int = 0) -> ctypes.CDLL:
    if mutant not in _libs:
        L = ctypes.CDLL(build(mutant))
        L.q4o_half_to_double.restype = ctypes.c_double
        L.q4o_half_to_double.argtypes = [ctypes.c_uint16]
        L.q4o_code.restype = ctypes.c_int
        L.q4o_code.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        L.q4o_gemv.restype = ctypes.c_int
        L.q4o_gemv.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        L.q4o_gemv_f64.restype = ctypes.c_int
        L.q4o_gemv_f64.argtypes = L.q4o_gemv.argtypes
        L.q4o_max_threads.restype = ctypes.c_int
        L.q8o_code.restype = ctypes.c_int
        L.q8o_code.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        for fn in (L.q8o_gemv, L.q8o_gemv_f64):
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        L.qbo_code.restype = ctypes.c_int
        L.qbo_code.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
        for fn in (L.qbo_gemv, L.qbo_gemv_f64):
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [ctypes.c_int] + [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        _libs[mutant] = L
    return _libs[mutant]


def max_threads() -> int:
    """OpenMP threads the C oracle uses (reported beside the CPU baseline).
    Infrastructure: no passage."""
    return _lib().q4o_max_threads()


def half_to_double(bits: int) -> float:
    """The C oracle's decoding of one IEEE binary16 bit pattern to fp64 (the fp16
    scales, biases and activations of the storage format; pinned against numpy on every
    pattern)."""
    return _lib().q4o_half_to_double(int(bits) & 0xFFFF)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def gemv(Wq, scales, biases, x, rows=None, nthreads: int = 0, mutant: int = 0):
    """y[M, R], A[M, R] in fp64 for W [N, K] (storage format) and x [M, K].

    x is fp16 (converted exactly) or fp64 (used as is).  ``rows`` (optional)
    selects output rows; R = len(rows) (else N).

    Follows BaseRT §3.3 (the matmul with the dequantisation inside its loop; w =
    scale*q + bias per 64-wide group) on the 4-bit files of MetalRT §2.1; the bit
    layout is the reading this library fixes (lowest nibble first).
    """
    Wq = np.ascontiguousarray(Wq, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.float16)
    biases = np.ascontiguousarray(biases, dtype=np.float16)
    x = np.atleast_2d(x)
    f64 = x.dtype == np.float64
    x = np.ascontiguousarray(x, dtype=np.float64 if f64 else np.float16)
    N, W = Wq.shape
    K = W * 8
    M = x.shape[0]
    if x.shape[1] != K or scales.shape != (N, K // 64) or biases.shape != (N, K // 64):
        raise ValueError("shape mismatch")
    if rows is None:
        R, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        if rows.size and (rows.min() < 0 or rows.max() >= N):
            raise ValueError("row out of range")
        R, rp = rows.size, _p(rows)
    y = np.empty((M, R), np.float64)
    A = np.empty((M, R), np.float64)
    if R == 0:
        return y, A
    L = _lib(mutant)
    fn = L.q4o_gemv_f64 if f64 else L.q4o_gemv
    xp = _p(x) if f64 else _p(x.view(np.uint16))
    rc = fn(_p(Wq), _p(scales.view(np.uint16)), _p(biases.view(np.uint16)), xp, M, N, K, rp, R, _p(y), _p(A),
            nthreads)
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return y, A


def gemv8(Wq, scales, biases, x, rows=None, nthreads: int = 0, mutant: int = 0):
    """gemv() for 8-bit codes: Wq uint32 [N, K/4], code k in byte k % 4 of
    word k // 4 (lowest byte first), q in 0..255, w = s * q + b per 64-group.

    Follows BaseRT §3.3 and §4.1 (one kernel per quantisation format; Q8 is one of the
    two evaluated).
    """
    Wq = np.ascontiguousarray(Wq, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.float16)
    biases = np.ascontiguousarray(biases, dtype=np.float16)
    x = np.atleast_2d(x)
    f64 = x.dtype == np.float64
    x = np.ascontiguousarray(x, dtype=np.float64 if f64 else np.float16)
    N, W = Wq.shape
    K = W * 4
    M = x.shape[0]
    if x.shape[1] != K or scales.shape != (N, K // 64) or biases.shape != (N, K // 64):
        raise ValueError("shape mismatch")
    if rows is None:
        R, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        if rows.size and (rows.min() < 0 or rows.max() >= N):
            raise ValueError("row out of range")
        R, rp = rows.size, _p(rows)
    y = np.empty((M, R), np.float64)
    A = np.empty((M, R), np.float64)
    if R == 0:
        return y, A
    L = _lib(mutant)
    fn = L.q8o_gemv_f64 if f64 else L.q8o_gemv
    xp = _p(x) if f64 else _p(x.view(np.uint16))
    rc = fn(_p(Wq), _p(scales.view(np.uint16)), _p(biases.view(np.uint16)), xp, M, N, K, rp, R, _p(y), _p(A),
            nthreads)
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return y, A


def gemvb(Wq, scales, biases, x, bits: int, rows=None, nthreads: int = 0, mutant: int = 0):
    """gemv() for b-bit codes (b in 2..8): Wq uint32 [N, K*b/32], code k of
    a row in bits b*k .. b*k+b-1 of the row's little-endian bit stream,
    q in 0..2^b-1, w = s * q + b per 64-group.

    Follows BaseRT §3.3 and §4.1 (kernels for 2- to 16-bit formats); the bit-stream
    layout is the reading this library fixes.
    """
    Wq = np.ascontiguousarray(Wq, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.float16)
    biases = np.ascontiguousarray(biases, dtype=np.float16)
    x = np.atleast_2d(x)
    f64 = x.dtype == np.float64
    x = np.ascontiguousarray(x, dtype=np.float64 if f64 else np.float16)
    N, W = Wq.shape
    K = W * 32 // bits
    M = x.shape[0]
    if W * 32 != K * bits or x.shape[1] != K or scales.shape != (N, K // 64) or biases.shape != (N, K // 64):
        raise ValueError("shape mismatch")
    if rows is None:
        R, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        if rows.size and (rows.min() < 0 or rows.max() >= N):
            raise ValueError("row out of range")
        R, rp = rows.size, _p(rows)
    y = np.empty((M, R), np.float64)
    A = np.empty((M, R), np.float64)
    if R == 0:
        return y, A
    L = _lib(mutant)
    fn = L.qbo_gemv_f64 if f64 else L.qbo_gemv
    xp = _p(x) if f64 else _p(x.view(np.uint16))
    rc = fn(_p(Wq), _p(scales.view(np.uint16)), _p(biases.view(np.uint16)), xp, M, N, K, bits, rp, R, _p(y), _p(A),
            nthreads)
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return y, A


def codeb(Wq_row, k: int, bits: int, mutant: int = 0) -> int:
    """The b-bit code k of one packed row (as the oracle reads it).

    Follows BaseRT §3.3 and §4.1 (b-bit formats), in the bit-stream reading.
    """
    row = np.ascontiguousarray(Wq_row, dtype=np.uint32)
    return _lib(mutant).qbo_code(_p(row), k, bits)


def code8(Wq_row, k: int, mutant: int = 0) -> int:
    """The 8-bit code k of one packed row (as the oracle reads it).

    Follows BaseRT §3.3 and §4.1 (the 8-bit format), lowest byte first.
    """
    row = np.ascontiguousarray(Wq_row, dtype=np.uint32)
    return _lib(mutant).q8o_code(_p(row), k)


def fp16(v) -> np.ndarray:
    """Round fp64 values to fp16, round-to-nearest-even (numpy converts
    directly from double, not through float32).

    The pages do not say how stored activations round; the reading taken is IEEE
    round-to-nearest-even, as the GPU's fp16 stores do.
    """
    return np.asarray(v, dtype=np.float64).astype(np.float16)


def silu(g):
    """SiLU(g) = g / (1 + exp(-g)) in fp64: the gate of the fused gate/up FFN step
    (BaseRT §3.3 fuses the FFN's operator sequence; the pages print no formula, this is
    the standard definition)."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def ulp16(v) -> np.ndarray:
    """Spacing of fp16 numbers at |v| (2^-24 in the subnormal range).

    Helper of the parity bar (an fp16 store may round either way of a value within the
    fp32 error). No passage.
    """
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


# ------------------------------------------------------------------ decode ---

DEFAULT_EPS = 1e-6


def rmsnorm(h, gamma=None, eps: float = DEFAULT_EPS):
    """h / sqrt(mean(h^2) + eps) * gamma, per row, in fp64 (gamma None = 1).

    Follows BaseRT §3.3 (normalisation kernels fused into the attention path and FFN)
    and MetalRT §5.1 (the norm kept in fp32); the RMS form is the reading taken for the
    pre-norm layer.
    """
    h = np.atleast_2d(np.asarray(h, dtype=np.float64))
    r = h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)
    if gamma is not None:
        r = r * np.asarray(gamma, dtype=np.float64)[None, :]
    return r


def _mat(m):
    return m.Wq, m.scales, m.biases


def decode_qkv(layer, h, rows=None, eps: float = DEFAULT_EPS):
    """q, k, v = W rmsnorm(h) for the fused QKV stage; dict of (y, A).

    Follows "Mac on-device AI performance breakthrough" §2.2 (Q, K, V merged into one
    product) and BaseRT §3.3 (the norm fused into the launch).
    """
    n = rmsnorm(h, layer.get("attn_norm"), eps)
    out = {}
    for nm in ("q", "k", "v"):
        r = None if rows is None else rows.get(nm)
        out[nm] = gemv(*_mat(layer[nm]), n, rows=r)
    return out


def decode_o(layer, a, h, rows=None):
    """h' = h + Wo a (fp64, before the fp16 store), A incl. |h|.

    Follows BaseRT §3 and §3.3 (the decode step as a chain of fused GEMVs; the residual
    add fused into the o launch) in the pre-norm dataflow reading.
    """
    y, A = gemv(*_mat(layer["o"]), a, rows=rows)
    hh = np.atleast_2d(h).astype(np.float64)
    if rows is not None:
        hh = hh[:, rows]
    return hh + y, A + np.abs(hh)


def decode_glu(layer, h, rows=None, eps: float = DEFAULT_EPS):
    """g, u from rmsnorm(h') and act = SiLU(g) * u (fp64, before the store).

    Follows BaseRT §3.3 (gate and up products with SiLU*up fused into one FFN launch).
    """
    n = rmsnorm(h, layer.get("ffn_norm"), eps)
    g, Ag = gemv(*_mat(layer["gate"]), n, rows=rows)
    u, Au = gemv(*_mat(layer["up"]), n, rows=rows)
    return g, Ag, u, Au, silu(g) * u


def decode_down(layer, act, h, rows=None):
    """h + Wd act for the down stage, fp64 before the fp16 store, and A including |h|
    (BaseRT §3.3: the FFN's operator sequence fused; the residual add is part of the
    dataflow reading)."""
    y, A = gemv(*_mat(layer["down"]), act, rows=rows)
    hh = np.atleast_2d(h).astype(np.float64)
    if rows is not None:
        hh = hh[:, rows]
    return hh + y, A + np.abs(hh)


def decode_logits(lm_head, h, final_norm=None, rows=None, eps: float = DEFAULT_EPS):
    """Wlm (rmsnorm(h) * final_norm): the last GEMV of the decode step (BaseRT §3: the
    decode hot path ends in the vocabulary projection; the final norm is part of the
    pre-norm reading)."""
    return gemv(*_mat(lm_head), rmsnorm(h, final_norm, eps), rows=rows)


def decode_layer(layer, h, eps: float = DEFAULT_EPS):
    """One layer, every stored activation rounded to fp16 as the GPU stores it.

    Follows BaseRT §3 (one decode layer as a fixed sequence of kernels) in the pre-norm
    dataflow reading.
    """
    qkv = decode_qkv(layer, h, eps=eps)
    q = fp16(qkv["q"][0])
    hm = fp16(decode_o(layer, q, h)[0])
    act = fp16(decode_glu(layer, hm, eps=eps)[4])
    ho = fp16(decode_down(layer, act, hm)[0])
    return {"q": q, "k": fp16(qkv["k"][0]), "v": fp16(qkv["v"][0]), "h_mid": hm, "act": act, "h": ho}


def decode_step(layers, lm_head, x, final_norm=None, eps: float = DEFAULT_EPS):
    """Whole decode step: fp16 x [M, hidden] -> fp64 logits [M, vocab].

    Follows BaseRT §3 and §3.1 (a whole decode step driven by a layer descriptor) in
    the pre-norm dataflow reading.
    """
    h = np.atleast_2d(x).astype(np.float16)
    for layer in layers:
        h = decode_layer(layer, h, eps)["h"]
    y, A = decode_logits(lm_head, h, final_norm, eps=eps)
    return y, A, h


def prefill_layer(layer, h, eps: float = DEFAULT_EPS):
    """One layer of the prefill stream (BaseRT §3.4 "Prefill": the prompt's
    tokens go through each matrix together).  The per-token dataflow of
    decode_layer, except that the two normalised activations are stored in
    fp16 before their matrix products (the tensor-core GEMM takes fp16
    operands); every stored activation is rounded to fp16 as the GPU stores it."""
    n = fp16(rmsnorm(h, layer.get("attn_norm"), eps))
    q = fp16(gemv(*_mat(layer["q"]), n)[0])
    k = fp16(gemv(*_mat(layer["k"]), n)[0])
    v = fp16(gemv(*_mat(layer["v"]), n)[0])
    hm = fp16(decode_o(layer, q, h)[0])
    n2 = fp16(rmsnorm(hm, layer.get("ffn_norm"), eps))
    g = gemv(*_mat(layer["gate"]), n2)[0]
    u = gemv(*_mat(layer["up"]), n2)[0]
    act = fp16(silu(g) * u)
    ho = fp16(decode_down(layer, act, hm)[0])
    return {"n": n, "q": q, "k": k, "v": v, "h_mid": hm, "n2": n2, "act": act, "h": ho}


def prefill(layers, lm_head, x, final_norm=None, eps: float = DEFAULT_EPS):
    """Prefill of T tokens: fp16 x [T, hidden] -> (final h [T, hidden] as
    fp16 values, logits y [1, vocab] and A of the LAST token).  The tokens do
    not interact in this stack (no attention), so chunking does not change
    the result; the logits come from the decode path's lm_head product.

    Follows BaseRT §3.4 (the prompt processed as GEMMs, chunk by chunk).
    """
    h = np.atleast_2d(x).astype(np.float16)
    for layer in layers:
        h = prefill_layer(layer, h, eps)["h"]
    y, A = decode_logits(lm_head, h[-1:], final_norm, eps=eps)
    return h, y, A


# ------------------------------------------------------- decode attention ---

DEFAULT_ROPE_THETA = 1.0e6


def rope(x, pos: int, head_dim: int, theta: float = DEFAULT_ROPE_THETA):
    """Rotary position embedding of every head of x [..., H*head_dim] at one
    position, rotate-half form: for i < d/2 the pair (x_i, x_{i+d/2}) turns by
    pos * theta^(-2i/d).  fp64.

    Follows BaseRT §3.3 (RoPE among the decode kernels); the pages print no formula, so
    the rotate-half form of Qwen3/Llama is the reading taken.
    """
    x = np.asarray(x, dtype=np.float64)
    d = head_dim
    xs = x.reshape(x.shape[:-1] + (-1, d))
    i = np.arange(d // 2, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / d)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = xs[..., : d // 2], xs[..., d // 2:]
    out = np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
    return out.reshape(x.shape)


def attention(q, k_cache, v_cache, n: int, head_dim: int, pos: int, theta: float = DEFAULT_ROPE_THETA,
              mutant: int = 0):
    """Decode attention of one token: q [Hq*d] (fp16 values, not yet rotated)
    against positions 0..n-1 of the caches [Hkv, max_seq, d] (keys stored
    rotated).  Query head h reads key/value head h // (Hq / Hkv).  Returns
    a [Hq*d] and A [Hq*d] = sum_j p_j |v_j| (fp64).

    Follows BaseRT §3.3 (attention among the decode kernels) and §3.2 (a preallocated
    KV cache); softmax(q.K^T / sqrt(d)).V is the plain definition.

    ``mutant`` plants a known mistake for the pin tests only (1: scores
    scaled by 1/d; 2: scores not scaled); 0 is the oracle.
    """
    d = head_dim
    qr = rope(q, pos, d, theta).reshape(-1, d)
    Hq, Hkv = qr.shape[0], k_cache.shape[0]
    g = Hq // Hkv
    a = np.empty((Hq, d))
    A = np.empty((Hq, d))
    scale = {0: np.sqrt(d), 1: float(d), 2: 1.0}[mutant]
    for h in range(Hq):
        K = k_cache[h // g, :n].astype(np.float64)
        V = v_cache[h // g, :n].astype(np.float64)
        s = K @ qr[h] / scale
        w = np.exp(s - s.max())
        w /= w.sum()
        a[h] = w @ V
        A[h] = w @ np.abs(V)
    return a.reshape(-1), A.reshape(-1)


def decode_layer_attn(layer, h, k_cache, v_cache, pos: int, head_dim: int, theta: float = DEFAULT_ROPE_THETA,
                      eps: float = DEFAULT_EPS):
    """decode_layer with attention in place of the stand-in a := q (BaseRT
    §3.3 lists RoPE and attention among the decode kernels): the new key
    (rotated) and value are written to position `pos` of the caches (fp16,
    in place), a = attention over positions 0..pos, rounded to fp16, feeds o."""
    qkv = decode_qkv(layer, h, eps=eps)
    q = fp16(qkv["q"][0])[0]
    k = fp16(qkv["k"][0])[0]
    v = fp16(qkv["v"][0])[0]
    Hkv = k_cache.shape[0]
    k_cache[:, pos] = fp16(rope(k, pos, head_dim, theta)).reshape(Hkv, head_dim)
    v_cache[:, pos] = v.reshape(Hkv, head_dim)
    a = fp16(attention(q, k_cache, v_cache, pos + 1, head_dim, pos, theta)[0])[None, :]
    hm = fp16(decode_o(layer, a, h)[0])
    act = fp16(decode_glu(layer, hm, eps=eps)[4])
    ho = fp16(decode_down(layer, act, hm)[0])
    return {"q": q, "k": k, "v": v, "a": a, "h_mid": hm, "act": act, "h": ho}


def decode_step_attn(layers, lm_head, x, caches, pos: int, head_dim: int, theta: float = DEFAULT_ROPE_THETA,
                     final_norm=None, eps: float = DEFAULT_EPS):
    """One decode step of one sequence with attention: x fp16 [1, hidden];
    caches = [(k_cache, v_cache)] per layer, updated at `pos`.  Returns
    (logits [1, vocab], A, final h).

    Follows BaseRT §3.2 and §3.3 (the decode step with its attention over the
    preallocated cache).
    """
    h = np.atleast_2d(x).astype(np.float16)
    for layer, (kc, vc) in zip(layers, caches):
        h = decode_layer_attn(layer, h, kc, vc, pos, head_dim, theta, eps)["h"]
    y, A = decode_logits(lm_head, h, final_norm, eps=eps)
    return y, A, h


def prefill_layer_attn(layer, h, k_cache, v_cache, pos0: int, head_dim: int, theta: float = DEFAULT_ROPE_THETA,
                       eps: float = DEFAULT_EPS):
    """prefill_layer with attention: tokens t = 0..T-1 sit at positions
    pos0 + t; their rotated keys and values are written to the caches (fp16),
    then token t attends over positions 0..pos0+t (causal), a rounded to fp16
    feeds o.  The normalised activations are stored in fp16 as in
    prefill_layer.

    Follows BaseRT §3.4 (prompt GEMMs) with causal attention over the cache (BaseRT
    §3.2, §3.3).
    """
    h = np.atleast_2d(h)
    T = h.shape[0]
    Hkv = k_cache.shape[0]
    n = fp16(rmsnorm(h, layer.get("attn_norm"), eps))
    q = fp16(gemv(*_mat(layer["q"]), n)[0])
    k = fp16(gemv(*_mat(layer["k"]), n)[0])
    v = fp16(gemv(*_mat(layer["v"]), n)[0])
    for t in range(T):
        k_cache[:, pos0 + t] = fp16(rope(k[t], pos0 + t, head_dim, theta)).reshape(Hkv, head_dim)
        v_cache[:, pos0 + t] = v[t].reshape(Hkv, head_dim)
    a = np.stack([fp16(attention(q[t], k_cache, v_cache, pos0 + t + 1, head_dim, pos0 + t, theta)[0])
                  for t in range(T)])
    hm = fp16(decode_o(layer, a, h)[0])
    n2 = fp16(rmsnorm(hm, layer.get("ffn_norm"), eps))
    g = gemv(*_mat(layer["gate"]), n2)[0]
    u = gemv(*_mat(layer["up"]), n2)[0]
    act = fp16(silu(g) * u)
    ho = fp16(decode_down(layer, act, hm)[0])
    return {"n": n, "q": q, "k": k, "v": v, "a": a, "h_mid": hm, "n2": n2, "act": act, "h": ho}


def prefill_attn(layers, lm_head, x, caches, pos0: int, head_dim: int, theta: float = DEFAULT_ROPE_THETA,
                 final_norm=None, eps: float = DEFAULT_EPS):
    """Prefill of T tokens at positions pos0.. with attention, filling the
    caches: (final h [T, hidden], logits y [1, vocab] and A of the last token).
    Chunking does not change the result (keys of earlier chunks are in the
    cache before later tokens attend to them).

    Follows BaseRT §3.4 (prefill in chunks) with the cache filled for the decode steps
    that follow (BaseRT §3.2).
    """
    h = np.atleast_2d(x).astype(np.float16)
    for layer, (kc, vc) in zip(layers, caches):
        h = prefill_layer_attn(layer, h, kc, vc, pos0, head_dim, theta, eps)["h"]
    y, A = decode_logits(lm_head, h[-1:], final_norm, eps=eps)
    return h, y, A


# --------------------------------------------------------------------- MoE ---

def moe_route(logits, topk: int):
    """Top-k routing of fp16 logits [T, E].

    Returns ids [T, topk] (by descending logit, ties to the lower expert),
    weights [T, topk] fp64 (softmax over the chosen logits), offsets [E+1],
    token_of [R], expert_of [R], rank_of [R] (R = T*topk rows sorted stably by
    (expert, token, rank)), pos [T, topk] (sorted row of each (t, k)).

    Follows BaseRT, abstract and Fig. 1 (MoE prefill on a Qwen3-30B-A3B-shaped model);
    the pages do not describe routing, so top-k with ties to the lower expert and a
    softmax over the chosen logits is the reading taken.
    """
    logits = np.asarray(logits, dtype=np.float16)
    T, E = logits.shape
    ids = np.empty((T, topk), np.int32)
    wts = np.empty((T, topk), np.float64)
    for t in range(T):
        vals = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-vals[e], e))[:topk]
        ids[t] = order
        chosen = np.array([vals[e] for e in order], np.float64)
        ex = np.exp(chosen - chosen.max())
        wts[t] = ex / ex.sum()
    triples = sorted((int(ids[t, k]), t, k) for t in range(T) for k in range(topk))
    R = T * topk
    token_of = np.empty(R, np.int32)
    expert_of = np.empty(R, np.int32)
    rank_of = np.empty(R, np.int32)
    pos = np.empty((T, topk), np.int32)
    counts = np.zeros(E, np.int64)
    for r, (e, t, k) in enumerate(triples):
        token_of[r], expert_of[r], rank_of[r] = t, e, k
        pos[t, k] = r
        counts[e] += 1
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    return {"ids": ids, "weights": wts, "offsets": offsets, "token_of": token_of,
            "expert_of": expert_of, "rank_of": rank_of, "pos": pos}


def _expert(m, e):
    return m.Wq[e], m.scales[e], m.biases[e]


def moe_gate_up_rows(gu, X_rows, experts, ffn: int):
    """For each row r: g = Wg[e] X_r, u = Wu[e] X_r (gate = rows 0..ffn-1 and up =
    rows ffn..2ffn-1 of the fused expert matrix).  Returns g, Ag, u, Au, act
    (fp64, before the fp16 store), each [len(rows), ffn].

    Follows BaseRT §3.4 (prefill GEMMs) on the routed experts of the abstract's MoE
    model.
    """
    n = len(experts)
    g = np.empty((n, ffn)); Ag = np.empty((n, ffn)); u = np.empty((n, ffn)); Au = np.empty((n, ffn))
    gate_rows = np.arange(ffn, dtype=np.int64)
    up_rows = gate_rows + ffn
    for i, e in enumerate(experts):
        W = _expert(gu, int(e))
        yg, ag = gemv(*W, X_rows[i:i + 1], rows=gate_rows)
        yu, au = gemv(*W, X_rows[i:i + 1], rows=up_rows)
        g[i], Ag[i], u[i], Au[i] = yg[0], ag[0], yu[0], au[0]
    return g, Ag, u, Au, silu(g) * u


def moe_down_rows(dn, H_rows, experts, cols=None):
    """Y_r = Wd[e] H_r for each row; returns (y, A) [len(rows), len(cols) or N].

    Follows BaseRT §3.4 (prefill GEMMs) on the routed experts of the abstract's MoE
    model.
    """
    out_y, out_a = [], []
    for i, e in enumerate(experts):
        y, A = gemv(*_expert(dn, int(e)), H_rows[i:i + 1], rows=cols)
        out_y.append(y[0]); out_a.append(A[0])
    return np.array(out_y), np.array(out_a)


def moe_combine(Y, pos, weights):
    """out[t] = sum_{k=0}^{topk-1} p[t,k] * Y[pos[t,k]], k in rank order, fp64.

    The weighted sum of the routed rows back per token; the pages do not describe it,
    so rank order in fp64 is the reading taken (BaseRT abstract: MoE prefill).
    """
    Y = np.asarray(Y, dtype=np.float64)
    T, topk = pos.shape
    out = np.zeros((T, Y.shape[1]))
    mag = np.zeros((T, Y.shape[1]))
    for t in range(T):
        for k in range(topk):
            out[t] += weights[t, k] * Y[pos[t, k]]
            mag[t] += np.abs(weights[t, k] * Y[pos[t, k]])
    return out, mag
