"""Seeded synthetic inputs for the Q4 group-64 decode matmul.

This module is shared by the tests, the benchmark and the smoke check. It only
draws random numbers and lays them out in the storage format; it holds none of
the arithmetic the library computes (no unpacking, no dequantisation, no dot
products), so the CUDA path and the CPU oracle both take their inputs from
here without sharing any computation.

Storage format (the affine "scale + bias per group" 4-bit format that the
MetalRT article's §2.1 benchmark files and the BaseRT paper's §3.3 kernels
consume; the pages do not print its bit layout, so this library fixes it):

* ``Wq``      uint32 ``[N, K/8]`` row-major.  Weight ``k`` of output row ``n``
  is the 4-bit code in word ``k // 8``, bits ``4*(k % 8)`` .. ``4*(k % 8)+3``
  (lowest nibble first).
* ``scales``  fp16 ``[N, K/64]`` row-major, one per 64-weight group.
* ``biases``  fp16 ``[N, K/64]`` row-major.
* the real weight is ``w = scale * q + bias`` with ``q`` in ``0..15``.

Recipe (all draws with numpy's PCG64 ``default_rng(seed)``):

* codes uniform in 0..15, independent.  Eight independent uniform nibbles
  packed into one word are exactly a uniform 32-bit word, so the words are
  drawn directly.
* ``scale = fp16(|N(0, 0.02)| / 7.5)`` (drawn in fp64, rounded once, RNE).
* ``bias  = -8 * scale`` from the fp16 scale (exact in fp16).
* activations ``x ~ N(0, 1)`` rounded to fp16; router logits likewise.

The 8-bit variant (``q8_matrix``) stores four codes per word, code ``k`` in
byte ``k % 4`` of word ``k // 4`` (lowest byte first), ``q`` in ``0..255``;
``scale = fp16(|N(0, 0.02)| / 127.5)``, ``bias = -128 * scale``.

The b-bit variant (``qb_matrix``, b in 2..8) packs the codes as a
little-endian bit stream per row: code k in bits b*k .. b*k+b-1 of the row
(crossing into the next uint32 when it must); ``scale = fp16(|N(0, 0.02)| /
((2^b - 1)/2))``, ``bias = -2^(b-1) * scale``.

Per-tensor seeds are ``BASE_SEED + index`` so every tensor of a model can be
regenerated alone (the oracle needs single matrices at full size).
"""
from __future__ import annotations

import dataclasses
import numpy as np

BASE_SEED = 1234
GROUP = 64          # weights per scale/bias group
CODES_PER_WORD = 8  # 4-bit codes per uint32


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


@dataclasses.dataclass
class Q4Matrix:
    """One Q4 matrix W[N, K] in storage format (host numpy arrays)."""
    Wq: np.ndarray       # uint32 [.., N, K/8]
    scales: np.ndarray   # float16 [.., N, K/64]
    biases: np.ndarray   # float16 [.., N, K/64]

    @property
    def N(self) -> int:
        return self.Wq.shape[-2]

    @property
    def K(self) -> int:
        return self.Wq.shape[-1] * CODES_PER_WORD

    def nbytes(self) -> int:
        return self.Wq.nbytes + self.scales.nbytes + self.biases.nbytes


def q4_matrix(seed: int, N: int, K: int, experts: int | None = None) -> Q4Matrix:
    """Random Q4 matrix (or a stack of ``experts`` of them) from one seed."""
    if K % GROUP:
        raise ValueError(f"K={K} is not a multiple of {GROUP}")
    lead = () if experts is None else (experts,)
    g = rng(seed)
    Wq = g.integers(0, 2**32, size=lead + (N, K // CODES_PER_WORD), dtype=np.uint32)
    s = (np.abs(g.standard_normal(size=lead + (N, K // GROUP)) * 0.02) / 7.5).astype(np.float16)
    b = (-8.0 * s.astype(np.float64)).astype(np.float16)
    return Q4Matrix(Wq, s, b)


def activations(seed: int, M: int, K: int) -> np.ndarray:
    """fp16 activations x[M, K] ~ N(0, 1)."""
    return rng(seed).standard_normal(size=(M, K)).astype(np.float16)


def router_logits(seed: int, T: int, E: int) -> np.ndarray:
    """fp16 router logits [T, E] ~ N(0, 1)."""
    return rng(seed).standard_normal(size=(T, E)).astype(np.float16)


# --------------------------------------------------------------------------
# Workload shapes.  Each decode layer is q, k, v, o, gate, up, down given as
# (N, K) = (outputs, inputs); y = W x.
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class DecodeShape:
    name: str
    n_layers: int
    hidden: int
    q: int        # q output width (= o input width)
    kv: int       # k/v output width
    ffn: int      # gate/up output width (= down input width)
    vocab: int

    def layer_linears(self):
        h = self.hidden
        return [("q", self.q, h), ("k", self.kv, h), ("v", self.kv, h),
                ("o", h, self.q), ("gate", self.ffn, h), ("up", self.ffn, h),
                ("down", h, self.ffn)]

    def weights_per_step(self) -> int:
        per_layer = sum(n * k for _, n, k in self.layer_linears())
        return self.n_layers * per_layer + self.vocab * self.hidden

    def weight_bytes_per_step(self) -> int:
        w = self.weights_per_step()
        return w // 2 + (w // GROUP) * 4


QWEN3_0P6B = DecodeShape("qwen3-0.6b-shaped", 28, 1024, 2048, 1024, 3072, 151936)
LLAMA32_3B = DecodeShape("llama-3.2-3b-shaped", 28, 3072, 3072, 1024, 8192, 128256)
QWEN3_4B = DecodeShape("qwen3-4b-shaped", 36, 2560, 4096, 1024, 9728, 151936)


def tiny_decode_shape(n_layers=3, hidden=256, q=384, kv=128, ffn=640, vocab=1000) -> DecodeShape:
    """A small model with the same structure, for tests the oracle finishes fast."""
    return DecodeShape("tiny", n_layers, hidden, q, kv, ffn, vocab)


def decode_weights(shape: DecodeShape, base_seed: int = BASE_SEED):
    """All matrices of a decode stack: list of per-layer dicts + lm_head.

    Seeds: layer l, linear j (order q,k,v,o,gate,up,down) uses
    base_seed + 16*l + j; lm_head uses base_seed + 16*n_layers.
    """
    layers = []
    for l in range(shape.n_layers):
        d = {}
        for j, (nm, N, K) in enumerate(shape.layer_linears()):
            d[nm] = q4_matrix(base_seed + 16 * l + j, N, K)
        layers.append(d)
    lm_head = q4_matrix(base_seed + 16 * shape.n_layers, shape.vocab, shape.hidden)
    return layers, lm_head


@dataclasses.dataclass
class Q8Matrix:
    """One matrix W[N, K] with 8-bit codes in storage format: ``Wq`` uint32
    ``[N, K/4]`` (code k in byte k % 4 of word k // 4, lowest byte first),
    fp16 ``scales`` and ``biases`` ``[N, K/64]``; ``w = scale * q + bias``."""
    Wq: np.ndarray
    scales: np.ndarray
    biases: np.ndarray

    @property
    def N(self) -> int:
        return self.Wq.shape[-2]

    @property
    def K(self) -> int:
        return self.Wq.shape[-1] * 4

    def nbytes(self) -> int:
        return self.Wq.nbytes + self.scales.nbytes + self.biases.nbytes


def q8_matrix(seed: int, N: int, K: int) -> Q8Matrix:
    """Random 8-bit matrix: codes uniform in 0..255 (four independent uniform
    bytes are a uniform word), scale = fp16(|N(0, 0.02)| / 127.5), bias =
    -128 * scale (exact in fp16), so w spans about the same range as the
    4-bit matrices."""
    if K % GROUP:
        raise ValueError(f"K={K} is not a multiple of {GROUP}")
    g = rng(seed)
    Wq = g.integers(0, 2**32, size=(N, K // 4), dtype=np.uint32)
    s = (np.abs(g.standard_normal((N, K // GROUP))) * 0.02 / 127.5).astype(np.float16)
    b = (-128.0 * s.astype(np.float64)).astype(np.float16)
    return Q8Matrix(Wq, s, b)


@dataclasses.dataclass
class QbMatrix:
    """One matrix W[N, K] with b-bit codes in storage format: ``Wq`` uint32
    ``[N, K*b/32]``, code k of a row in bits b*k .. b*k+b-1 of the row's
    little-endian bit stream (a code may cross into the next word); fp16
    ``scales`` and ``biases`` ``[N, K/64]``; ``w = scale * q + bias``.
    ``codes`` keeps the drawn codes [N, K] (test input, not read by the
    library or the oracle)."""
    Wq: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    bits: int
    codes: np.ndarray

    @property
    def N(self) -> int:
        return self.Wq.shape[-2]

    @property
    def K(self) -> int:
        return self.Wq.shape[-1] * 32 // self.bits

    def nbytes(self) -> int:
        return self.Wq.nbytes + self.scales.nbytes + self.biases.nbytes


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes [N, K] (each < 2^bits) into uint32 words [N, K*bits/32],
    code k at bits bits*k .. of the row's little-endian bit stream."""
    N, K = codes.shape
    if (K * bits) % 32:
        raise ValueError("K * bits is not a multiple of 32")
    c = codes.astype(np.uint32)
    bitarr = ((c[:, :, None] >> np.arange(bits, dtype=np.uint32)[None, None, :]) & 1).astype(np.uint8)
    packed = np.packbits(bitarr.reshape(N, K * bits), axis=1, bitorder="little")
    return np.ascontiguousarray(packed).view("<u4").astype(np.uint32)


def qb_matrix(seed: int, N: int, K: int, bits: int) -> QbMatrix:
    """Random b-bit matrix: codes uniform in 0..2^b-1, scale =
    fp16(|N(0, 0.02)| / ((2^b - 1) / 2)), bias = -2^(b-1) * scale (exact in
    fp16), so w spans about the same range as the 4-bit matrices."""
    if K % GROUP:
        raise ValueError(f"K={K} is not a multiple of {GROUP}")
    g = rng(seed)
    codes = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint32)
    s = (np.abs(g.standard_normal((N, K // GROUP))) * 0.02 / ((2 ** bits - 1) / 2)).astype(np.float16)
    b = (-(2.0 ** (bits - 1)) * s.astype(np.float64)).astype(np.float16)
    return QbMatrix(pack_codes(codes, bits), s, b, bits, codes)


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    hidden: int
    experts: int
    ffn: int      # per-expert gate/up width (= down input width)
    topk: int


QWEN3_30B_A3B_MOE = MoEShape("qwen3-30b-a3b-moe-layer", 2048, 128, 768, 8)


def moe_weights(shape: MoEShape, base_seed: int = BASE_SEED + 9000):
    """Expert stacks: gate/up fused as [E, 2*ffn, hidden/8] (rows 0..ffn-1 gate,
    ffn..2ffn-1 up) and down as [E, hidden, ffn/8]."""
    gu = q4_matrix(base_seed + 0, 2 * shape.ffn, shape.hidden, experts=shape.experts)
    dn = q4_matrix(base_seed + 1, shape.hidden, shape.ffn, experts=shape.experts)
    return gu, dn
