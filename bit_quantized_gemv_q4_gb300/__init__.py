"""Python binding of the Q4 group-64 decode-matmul library (``include/q4.h``).

Argument marshalling only: every function here forwards to the C ABI of
``libq4gb300.so``; each step of the computation runs in the library's CUDA
kernels.  torch tensors are accepted for device buffers (their data pointers
are passed) and the current torch stream is used unless one is given.  There
is no fallback: if the library is missing or a call fails, an exception is
raised.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "Q4Error", "lib", "q4_selftest_expired_wait", "q4_gemv", "q4_gemv8", "q4_gemv_ex", "Segment", "q4_device_status",
    "LayerTable", "q4_decode_step", "q4_decode_workspace_bytes", "q4_decode_buffers",
    "q4_layer_table_release", "q4_decode_path", "q4_moe_route", "q4_moe_route_workspace_bytes",
    "q4_moe_gather", "q4_moe_gemm", "q4_moe_combine",
    "Q4_F32", "Q4_F16", "Q4_GEMV_PLAIN", "Q4_GEMV_GLU", "Q4_DECODE_NO_GRAPH", "Q4_DECODE_NO_PDL",
    "Q4_DECODE_TAGGED",
    "Q4_DECODE_PERSISTENT", "Q4_DECODE_CLUSTERED", "Q4_GEMV_EARLY_WEIGHTS",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libq4gb300.so")

Q4_F32, Q4_F16 = 0, 1
Q4_GEMV_PLAIN, Q4_GEMV_GLU = 0, 1
Q4_DECODE_NO_GRAPH, Q4_DECODE_NO_PDL, Q4_DECODE_TAGGED, Q4_DECODE_PERSISTENT = 1, 2, 4, 8
Q4_DECODE_ATTENTION = 16
Q4_DECODE_CLUSTERED = 32
Q4_GEMV_EARLY_WEIGHTS = 1
Q4_MAX_SEGMENTS = 4

STATUS = {0: "Q4_OK", -1: "Q4_ERR_INVALID_ARG", -2: "Q4_ERR_UNSUPPORTED", -3: "Q4_ERR_MISALIGNED",
          -4: "Q4_ERR_CUDA", -5: "Q4_ERR_TIMEOUT", -6: "Q4_ERR_NO_DEVICE", -7: "Q4_ERR_DEVICE_CHECK"}

# Every symbol include/q4.h declares.
EXPORTS = ["q4_last_error", "q4_status_string", "q4_version", "q4_device_status",
           "q4_selftest_expired_wait", "q4_gemv", "q4_gemv8", "q4_gemv_bits",
           "q4_gemv_ex", "q4_decode_workspace_bytes", "q4_decode_buffers", "q4_decode_step",
           "q4_layer_table_release", "q4_decode_path", "q4_moe_route_workspace_bytes", "q4_moe_route",
           "q4_moe_route_noalloc",
           "q4_moe_gather", "q4_moe_gemm", "q4_moe_combine", "q4_gemm", "q4_prefill_workspace_bytes",
           "q4_prefill", "q4_attention_workspace_bytes", "q4_attention", "q4_gemm_workspace_bytes",
           "q4_prefill_buffers"]


class Q4Error(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {text}")


vp = ctypes.c_void_p
i32 = ctypes.c_int


class q4_segment(ctypes.Structure):
    _fields_ = [("Wq", vp), ("scales", vp), ("biases", vp), ("N", i32), ("ldy", i32), ("y", vp),
                ("residual", vp)]


class q4_gemv_desc(ctypes.Structure):
    _fields_ = [("M", i32), ("K", i32), ("x", vp), ("ldx", i32), ("n_segments", i32),
                ("seg", q4_segment * Q4_MAX_SEGMENTS), ("out_dtype", i32), ("mode", i32), ("x_rmsnorm", i32),
                ("norm_weight", vp), ("norm_eps", ctypes.c_float), ("flags", i32)]


class q4_linear(ctypes.Structure):
    _fields_ = [("Wq", vp), ("scales", vp), ("biases", vp), ("N", i32), ("K", i32)]


class q4_layer_weights(ctypes.Structure):
    _fields_ = [(n, q4_linear) for n in ("q", "k", "v", "o", "gate", "up", "down")] + [
        ("attn_norm", vp), ("ffn_norm", vp), ("k_cache", vp), ("v_cache", vp)]


class q4_layer_table(ctypes.Structure):
    _fields_ = [("n_layers", i32), ("hidden", i32), ("M", i32), ("layers", ctypes.POINTER(q4_layer_weights)),
                ("lm_head", q4_linear), ("final_norm", vp), ("norm_eps", ctypes.c_float),
                ("logits_dtype", i32), ("workspace", vp),
                ("workspace_bytes", ctypes.c_size_t), ("flags", i32), ("plan", vp),
                ("head_dim", i32), ("max_seq", i32), ("rope_theta", ctypes.c_float), ("pos", vp)]


class q4_decode_buffers_t(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("h", "h_mid", "q", "k", "v", "act", "a")]


class q4_moe_desc(ctypes.Structure):
    _fields_ = [("E", i32), ("N", i32), ("K", i32), ("R", i32), ("mode", i32), ("out_dtype", i32)]


class q4_attention_desc(ctypes.Structure):
    _fields_ = [("q", vp), ("k", vp), ("v", vp), ("k_cache", vp), ("v_cache", vp), ("pos", vp),
                ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32), ("max_seq", i32),
                ("rope_theta", ctypes.c_float), ("a", vp), ("workspace", vp), ("workspace_bytes", ctypes.c_size_t)]


class q4_prefill_buffers_t(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("n", "q", "k", "v", "act", "a")]


class q4_gemm_desc(ctypes.Structure):
    _fields_ = [("M", i32), ("X", vp), ("w", q4_linear), ("up", q4_linear), ("mode", i32), ("out_dtype", i32),
                ("Y", vp), ("residual", vp), ("workspace", vp), ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libq4gb300.so`` (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run bit_quantized_gemv_q4_gb300/build.py "
                              "(or __graft_entry__.build()) first")
        L = ctypes.CDLL(LIB_PATH)
        st = ctypes.c_int
        L.q4_last_error.restype = ctypes.c_char_p
        L.q4_status_string.restype = ctypes.c_char_p
        L.q4_status_string.argtypes = [st]
        L.q4_version.restype = i32
        L.q4_device_status.restype = st
        L.q4_device_status.argtypes = [vp]
        L.q4_selftest_expired_wait.restype = st
        L.q4_selftest_expired_wait.argtypes = [vp]
        L.q4_gemv.restype = st
        L.q4_gemv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
        L.q4_gemv8.restype = st
        L.q4_gemv8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
        L.q4_gemv_bits.restype = st
        L.q4_gemv_bits.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
        L.q4_gemv_ex.restype = st
        L.q4_gemv_ex.argtypes = [ctypes.POINTER(q4_gemv_desc), vp]
        L.q4_decode_workspace_bytes.restype = ctypes.c_size_t
        L.q4_decode_workspace_bytes.argtypes = [ctypes.POINTER(q4_layer_table)]
        L.q4_decode_buffers.restype = st
        L.q4_decode_buffers.argtypes = [ctypes.POINTER(q4_layer_table), ctypes.POINTER(q4_decode_buffers_t)]
        L.q4_decode_step.restype = st
        L.q4_decode_step.argtypes = [ctypes.POINTER(q4_layer_table), vp, vp, vp]
        L.q4_layer_table_release.restype = st
        L.q4_layer_table_release.argtypes = [ctypes.POINTER(q4_layer_table)]
        L.q4_decode_path.restype = ctypes.c_int
        L.q4_decode_path.argtypes = [ctypes.POINTER(q4_layer_table)]
        L.q4_moe_route_workspace_bytes.restype = ctypes.c_size_t
        L.q4_moe_route_workspace_bytes.argtypes = [i32, i32, i32]
        L.q4_moe_route.restype = st
        L.q4_moe_route.argtypes = [vp, i32, i32, i32] + [vp] * 7 + [ctypes.c_size_t, vp]
        L.q4_moe_route_noalloc.restype = st
        L.q4_moe_route_noalloc.argtypes = [vp, i32, i32, i32] + [vp] * 6 + [vp]
        L.q4_moe_gather.restype = st
        L.q4_moe_gather.argtypes = [vp, i32, i32, vp, i32, vp, vp]
        L.q4_moe_gemm.restype = st
        L.q4_moe_gemm.argtypes = [vp] * 7 + [ctypes.POINTER(q4_moe_desc), vp]
        L.q4_moe_combine.restype = st
        L.q4_moe_combine.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, i32, vp]
        L.q4_gemm_workspace_bytes.restype = ctypes.c_size_t
        L.q4_gemm_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.q4_gemm.restype = st
        L.q4_gemm.argtypes = [ctypes.POINTER(q4_gemm_desc), vp]
        L.q4_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.q4_prefill_workspace_bytes.argtypes = [ctypes.POINTER(q4_layer_table), i32]
        L.q4_prefill.restype = st
        L.q4_prefill.argtypes = [ctypes.POINTER(q4_layer_table), vp, i32, i32, vp, vp, ctypes.c_size_t, vp]
        L.q4_prefill_buffers.restype = st
        L.q4_prefill_buffers.argtypes = [ctypes.POINTER(q4_layer_table), i32, vp, ctypes.POINTER(q4_prefill_buffers_t)]
        L.q4_attention_workspace_bytes.restype = ctypes.c_size_t
        L.q4_attention_workspace_bytes.argtypes = [i32, i32, i32]
        L.q4_attention.restype = st
        L.q4_attention.argtypes = [ctypes.POINTER(q4_attention_desc), vp]
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise Q4Error(status, where, lib().q4_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    """Device pointer of a torch tensor in CUDA memory, an int (a raw device
    pointer, passed as is), or None.  A tensor in host memory is refused here:
    the kernels would dereference its address on the device."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"expected a tensor in CUDA device memory, got one on {t.device}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def q4_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device error status (0 = ok)."""
    return lib().q4_device_status(_stream(stream))


def q4_selftest_expired_wait(stream=None):
    """Enqueue the bounded-wait self-test (each wait expires after 2 s)."""
    _check(lib().q4_selftest_expired_wait(_stream(stream)), "q4_selftest_expired_wait")


# ------------------------------------------------------------------ GEMV ---

def q4_gemv(Wq, scales, biases, x, y, M: int, N: int, K: int, stream=None):
    _check(lib().q4_gemv(_ptr(Wq), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K, _stream(stream)),
           "q4_gemv")


def q4_gemv8(Wq, scales, biases, x, y, M: int, N: int, K: int, stream=None):
    """q4_gemv for 8-bit codes: Wq uint32 [N, K/4], lowest byte first."""
    _check(lib().q4_gemv8(_ptr(Wq), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K, _stream(stream)),
           "q4_gemv8")


def q4_gemv_bits(Wq, scales, biases, x, y, M: int, N: int, K: int, bits: int, stream=None):
    """q4_gemv for b-bit codes (b in 2, 3, 4, 5, 6, 8): Wq uint32 [N, K*b/32],
    a little-endian bit stream per row."""
    _check(lib().q4_gemv_bits(_ptr(Wq), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K, bits,
                              _stream(stream)), "q4_gemv_bits")


class Segment:
    """One matrix of a fused launch: weights, output, optional fp16 residual."""

    def __init__(self, Wq, scales, biases, N: int, y=None, residual=None, ldy: int = 0):
        self.Wq, self.scales, self.biases, self.N, self.y, self.residual, self.ldy = (
            Wq, scales, biases, N, y, residual, ldy)


def q4_gemv_ex(segments, x, M: int, K: int, out_dtype=Q4_F32, mode=Q4_GEMV_PLAIN, ldx: int = 0,
               rmsnorm: bool = False, norm_weight=None, norm_eps: float = 1e-6, stream=None, flags: int = 0):
    d = q4_gemv_desc()
    d.flags = flags
    d.M, d.K, d.x, d.ldx = M, K, _ptr(x), ldx
    d.x_rmsnorm, d.norm_weight, d.norm_eps = int(rmsnorm), _ptr(norm_weight), norm_eps
    d.n_segments = len(segments)
    for i, s in enumerate(segments):
        d.seg[i] = q4_segment(_ptr(s.Wq), _ptr(s.scales), _ptr(s.biases), s.N, s.ldy, _ptr(s.y),
                              _ptr(s.residual))
    d.out_dtype, d.mode = out_dtype, mode
    _check(lib().q4_gemv_ex(ctypes.byref(d), _stream(stream)), "q4_gemv_ex")


# ---------------------------------------------------------------- decode ---

def _linear(Wq, scales, biases, N, K) -> q4_linear:
    return q4_linear(_ptr(Wq), _ptr(scales), _ptr(biases), N, K)


class LayerTable:
    """Owns a ``q4_layer_table`` and keeps the tensors it points to alive.

    ``layers``: list of dicts name -> (Wq, scales, biases, N, K) for q, k, v,
    o, gate, up, down, and optionally "attn_norm" / "ffn_norm" -> fp16 [hidden]
    device tensors; ``lm_head`` likewise; ``final_norm`` optional."""

    def __init__(self, layers, lm_head, hidden: int, M: int, workspace=None, workspace_bytes: int = 0,
                 logits_dtype=Q4_F32, flags: int = 0, final_norm=None, norm_eps: float = 0.0,
                 head_dim: int = 0, max_seq: int = 0, rope_theta: float = 1.0e6, pos=None):
        self._keep = (layers, lm_head, workspace, final_norm, pos)
        n = len(layers)
        self._arr = (q4_layer_weights * max(n, 1))()
        for i, d in enumerate(layers):
            for nm in ("q", "k", "v", "o", "gate", "up", "down"):
                setattr(self._arr[i], nm, _linear(*d[nm]))
            self._arr[i].attn_norm = _ptr(d.get("attn_norm"))
            self._arr[i].ffn_norm = _ptr(d.get("ffn_norm"))
            self._arr[i].k_cache = _ptr(d.get("k_cache"))
            self._arr[i].v_cache = _ptr(d.get("v_cache"))
        t = q4_layer_table()
        t.n_layers, t.hidden, t.M = n, hidden, M
        t.layers = ctypes.cast(self._arr, ctypes.POINTER(q4_layer_weights))
        t.lm_head = _linear(*lm_head)
        t.final_norm, t.norm_eps = _ptr(final_norm), norm_eps
        t.logits_dtype, t.flags = logits_dtype, flags
        t.workspace, t.workspace_bytes = _ptr(workspace), workspace_bytes
        t.plan = None
        t.head_dim, t.max_seq, t.rope_theta, t.pos = head_dim, max_seq, rope_theta, _ptr(pos)
        self.t = t

    def set_workspace(self, workspace, nbytes: int):
        self._keep = self._keep[:2] + (workspace,) + self._keep[3:]
        self.t.workspace, self.t.workspace_bytes = _ptr(workspace), nbytes

    def release(self):
        q4_layer_table_release(self)

    def __del__(self):
        try:
            if self.t.plan:
                lib().q4_layer_table_release(ctypes.byref(self.t))
        except Exception:
            pass


def q4_decode_workspace_bytes(table: LayerTable) -> int:
    n = lib().q4_decode_workspace_bytes(ctypes.byref(table.t))
    if n == 0:
        raise Q4Error(-1, "q4_decode_workspace_bytes", lib().q4_last_error().decode())
    return n


def q4_decode_buffers(table: LayerTable) -> dict:
    b = q4_decode_buffers_t()
    _check(lib().q4_decode_buffers(ctypes.byref(table.t), ctypes.byref(b)), "q4_decode_buffers")
    return {n: getattr(b, n) for n in ("h", "h_mid", "q", "k", "v", "act", "a")}


def q4_decode_step(table: LayerTable, x, logits, stream=None):
    _check(lib().q4_decode_step(ctypes.byref(table.t), _ptr(x), _ptr(logits), _stream(stream)), "q4_decode_step")


def q4_decode_path(table: LayerTable) -> int:
    """0 = not planned, 1 = per-stage launches, 2 = persistent launch, 3 = clustered step + lm_head."""
    return lib().q4_decode_path(ctypes.byref(table.t))


def q4_layer_table_release(table: LayerTable):
    _check(lib().q4_layer_table_release(ctypes.byref(table.t)), "q4_layer_table_release")


# ------------------------------------------------------------------- MoE ---

def q4_moe_route_workspace_bytes(T: int, E: int, topk: int) -> int:
    return lib().q4_moe_route_workspace_bytes(T, E, topk)


def q4_moe_route(logits, T, E, topk, topk_ids, topk_weights, offsets, token_of, expert_of, pos, workspace,
                 workspace_bytes, stream=None):
    _check(lib().q4_moe_route(_ptr(logits), T, E, topk, _ptr(topk_ids), _ptr(topk_weights), _ptr(offsets),
                              _ptr(token_of), _ptr(expert_of), _ptr(pos), _ptr(workspace), workspace_bytes,
                              _stream(stream)), "q4_moe_route")


def q4_moe_route_noalloc(logits, T, E, topk, topk_ids, topk_weights, offsets, token_of, expert_of, pos,
                         stream=None):
    """q4_moe_route with the library's static scratch instead of a workspace."""
    _check(lib().q4_moe_route_noalloc(_ptr(logits), T, E, topk, _ptr(topk_ids), _ptr(topk_weights), _ptr(offsets),
                                      _ptr(token_of), _ptr(expert_of), _ptr(pos), _stream(stream)),
           "q4_moe_route_noalloc")


def q4_moe_gather(X, T, K, token_of, R, X_sorted, stream=None):
    _check(lib().q4_moe_gather(_ptr(X), T, K, _ptr(token_of), R, _ptr(X_sorted), _stream(stream)),
           "q4_moe_gather")


def q4_moe_gemm(Wq, scales, biases, X, expert_ids, offsets, Y, E, N, K, R, mode=Q4_GEMV_PLAIN,
                out_dtype=Q4_F32, stream=None):
    d = q4_moe_desc(E, N, K, R, mode, out_dtype)
    _check(lib().q4_moe_gemm(_ptr(Wq), _ptr(scales), _ptr(biases), _ptr(X), _ptr(expert_ids), _ptr(offsets),
                             _ptr(Y), ctypes.byref(d), _stream(stream)), "q4_moe_gemm")


def q4_moe_combine(Y, y_dtype, N, pos, topk_weights, T, topk, out, out_dtype, stream=None):
    _check(lib().q4_moe_combine(_ptr(Y), y_dtype, N, _ptr(pos), _ptr(topk_weights), T, topk, _ptr(out),
                                out_dtype, _stream(stream)), "q4_moe_combine")


# --------------------------------------------------------------- prefill ---

def q4_gemm_workspace_bytes(M: int, N: int, K: int, mode=Q4_GEMV_PLAIN) -> int:
    return lib().q4_gemm_workspace_bytes(M, N, K, mode)


def q4_gemm(w, X, Y, M: int, mode=Q4_GEMV_PLAIN, out_dtype=Q4_F32, up=None, residual=None, workspace=None,
            workspace_bytes: int = 0, stream=None):
    """Dense Y[M, N] = X[M, K] W^T on the tensor cores.  ``w`` (and ``up`` in
    GLU mode) are (Wq, scales, biases, N, K); a workspace lets K split."""
    d = q4_gemm_desc()
    d.M, d.X, d.w = M, _ptr(X), _linear(*w)
    if up is not None:
        d.up = _linear(*up)
    d.mode, d.out_dtype, d.Y, d.residual = mode, out_dtype, _ptr(Y), _ptr(residual)
    d.workspace, d.workspace_bytes = _ptr(workspace), workspace_bytes
    _check(lib().q4_gemm(ctypes.byref(d), _stream(stream)), "q4_gemm")


def q4_prefill_workspace_bytes(table: LayerTable, chunk: int) -> int:
    n = lib().q4_prefill_workspace_bytes(ctypes.byref(table.t), chunk)
    if n == 0:
        raise Q4Error(-1, "q4_prefill_workspace_bytes", lib().q4_last_error().decode())
    return n


def q4_prefill(table: LayerTable, h, T: int, chunk: int, logits, workspace, workspace_bytes: int, stream=None):
    """Chunked prefill: h fp16 [T, hidden] in place; logits of the last token (or None)."""
    _check(lib().q4_prefill(ctypes.byref(table.t), _ptr(h), T, chunk, _ptr(logits), _ptr(workspace),
                            workspace_bytes, _stream(stream)), "q4_prefill")


# ------------------------------------------------------------- attention ---

def q4_attention_workspace_bytes(n_q_heads: int, head_dim: int, max_seq: int) -> int:
    return lib().q4_attention_workspace_bytes(n_q_heads, head_dim, max_seq)


def q4_attention(q, k, v, k_cache, v_cache, pos, n_q_heads: int, n_kv_heads: int, head_dim: int, max_seq: int,
                 a, workspace, workspace_bytes: int, rope_theta: float = 1.0e6, stream=None):
    """One token's cache append and decode attention (pos: device int32, not advanced)."""
    d = q4_attention_desc(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(pos), n_q_heads,
                          n_kv_heads, head_dim, max_seq, rope_theta, _ptr(a), _ptr(workspace), workspace_bytes)
    _check(lib().q4_attention(ctypes.byref(d), _stream(stream)), "q4_attention")


def q4_prefill_buffers(table: LayerTable, chunk: int, workspace) -> dict:
    b = q4_prefill_buffers_t()
    _check(lib().q4_prefill_buffers(ctypes.byref(table.t), chunk, _ptr(workspace), ctypes.byref(b)),
           "q4_prefill_buffers")
    return {n: getattr(b, n) for n in ("n", "q", "k", "v", "act", "a")}
