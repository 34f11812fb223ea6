"""C ABI checks that need no GPU: the library loads, exports every function
include/q4.h declares, its structs have the layout the Python binding uses,
and host-side argument validation rejects bad calls before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

import bit_quantized_gemv_q4_gb300 as q4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return q4.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_[a-z0-9_]+)\s*\(", text)) - {"q4_status"})


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(q4.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", q4.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    for f in declared_functions():
        assert hasattr(L, f)


def test_version_and_status_strings(L):
    assert L.q4_version() == 100
    assert L.q4_status_string(0) == b"ok"
    assert L.q4_status_string(-3).startswith(b"misaligned")
    assert L.q4_status_string(-5).startswith(b"device-side wait")


def test_struct_layouts_match_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "q4.h"
#define P(T) printf(#T " %zu\\n", sizeof(T));
#define O(T, f) printf(#T "." #f " %zu\\n", offsetof(T, f));
int main(void) {
  P(q4_segment) P(q4_gemv_desc) P(q4_linear) P(q4_layer_weights) P(q4_layer_table)
  P(q4_decode_buffers_t) P(q4_moe_desc) P(q4_gemm_desc)
  O(q4_gemm_desc, X) O(q4_gemm_desc, w) O(q4_gemm_desc, up) O(q4_gemm_desc, mode) O(q4_gemm_desc, Y)
  O(q4_gemm_desc, residual) O(q4_gemm_desc, workspace_bytes) P(q4_attention_desc) O(q4_attention_desc, rope_theta) O(q4_attention_desc, a)
  O(q4_attention_desc, workspace_bytes) O(q4_layer_weights, k_cache) O(q4_layer_weights, v_cache)
  O(q4_layer_table, head_dim) O(q4_layer_table, rope_theta) O(q4_layer_table, pos) O(q4_decode_buffers_t, a)
  P(q4_prefill_buffers_t) O(q4_prefill_buffers_t, a)
  O(q4_gemv_desc, seg) O(q4_gemv_desc, out_dtype) O(q4_gemv_desc, mode)
  O(q4_segment, y) O(q4_segment, residual)
  O(q4_layer_table, layers) O(q4_layer_table, lm_head) O(q4_layer_table, workspace)
  O(q4_layer_table, workspace_bytes) O(q4_layer_table, flags) O(q4_layer_table, plan)
  O(q4_layer_weights, down) O(q4_layer_weights, ffn_norm) O(q4_moe_desc, out_dtype)
  O(q4_gemv_desc, x_rmsnorm) O(q4_gemv_desc, norm_weight) O(q4_gemv_desc, norm_eps) O(q4_gemv_desc, flags)
  O(q4_layer_table, final_norm) O(q4_layer_table, norm_eps) O(q4_layer_table, logits_dtype)
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(ln.rsplit(" ", 1) for ln in subprocess.run([str(exe)], capture_output=True, text=True,
                                                          check=True).stdout.split("\n") if ln)
    S = {"q4_segment": q4.q4_segment, "q4_gemv_desc": q4.q4_gemv_desc, "q4_linear": q4.q4_linear,
         "q4_layer_weights": q4.q4_layer_weights, "q4_layer_table": q4.q4_layer_table,
         "q4_decode_buffers_t": q4.q4_decode_buffers_t, "q4_moe_desc": q4.q4_moe_desc,
         "q4_gemm_desc": q4.q4_gemm_desc, "q4_attention_desc": q4.q4_attention_desc,
         "q4_prefill_buffers_t": q4.q4_prefill_buffers_t}
    for key, val in got.items():
        if "." in key:
            t, f = key.split(".")
            assert getattr(S[t], f).offset == int(val), key
        else:
            assert ctypes.sizeof(S[key]) == int(val), key


# Host-side validation runs before any CUDA call, so these need no GPU.  The
# pointers are never dereferenced.
FAKE = 0x10000


@pytest.mark.parametrize("M,N,K,expect", [(0, 8, 64, -1), (9, 8, 64, -2), (1, 0, 64, -1), (1, 8, 100, -1),
                                          (1, 8, 0, -1), (1, 8, -64, -1)])
def test_gemv_rejects_bad_sizes(L, M, N, K, expect):
    assert L.q4_gemv(FAKE, FAKE, FAKE, FAKE, FAKE, M, N, K, None) == expect
    assert L.q4_last_error() != b""


def test_gemv_bits_refusals(L):
    for bits, M, want in ((7, 1, -1), (1, 1, -1), (9, 1, -1), (3, 2, -2), (6, 4, -2)):
        assert L.q4_gemv_bits(FAKE, FAKE, FAKE, FAKE, FAKE, M, 8, 64, bits, None) == want, (bits, M)


def test_gemv_rejects_null_and_misaligned(L):
    assert L.q4_gemv(None, FAKE, FAKE, FAKE, FAKE, 1, 8, 64, None) == -1
    assert L.q4_gemv(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 1, 8, 64, None) == -3
    assert L.q4_gemv(FAKE, FAKE, FAKE, FAKE + 2, FAKE, 1, 8, 64, None) == -3


def test_gemv_ex_rejects_bad_descriptors(L):
    d = q4.q4_gemv_desc()
    d.M, d.K, d.x, d.n_segments = 1, 64, FAKE, 2
    for i in range(2):
        d.seg[i] = q4.q4_segment(FAKE, FAKE, FAKE, 8, 0, FAKE, None)
    d.mode = q4.Q4_GEMV_GLU
    d.out_dtype = q4.Q4_F32
    assert L.q4_gemv_ex(ctypes.byref(d), None) == -1      # GLU writes fp16
    d.out_dtype = q4.Q4_F16
    d.seg[1].N = 16
    assert L.q4_gemv_ex(ctypes.byref(d), None) == -1      # GLU widths differ
    d.mode = q4.Q4_GEMV_PLAIN
    d.n_segments = 5
    assert L.q4_gemv_ex(ctypes.byref(d), None) == -1
    d.n_segments = 1
    d.ldx = 12
    assert L.q4_gemv_ex(ctypes.byref(d), None) == -1      # ldx < K
    d.ldx = 68
    assert L.q4_gemv_ex(ctypes.byref(d), None) == -3      # ldx % 8
    d.ldx = 0
    d.out_dtype = q4.Q4_F32
    d.seg[0].residual = FAKE
    assert L.q4_gemv_ex(ctypes.byref(d), None) == -1      # residual needs fp16 out
    assert L.q4_gemv_ex(None, None) == -1


def lin(N, K, p=FAKE):
    return (p, p, p, N, K)


def test_decode_table_validation_and_workspace(L):
    layer = {"q": lin(128, 64), "k": lin(64, 64), "v": lin(64, 64), "o": lin(64, 128), "gate": lin(192, 64),
             "up": lin(192, 64), "down": lin(64, 192)}
    t = q4.LayerTable([layer, layer], lin(100, 64), hidden=64, M=2)
    n = q4.q4_decode_workspace_bytes(t)
    # plain fp16: h, h_mid 2*64*2 B each; q 2*128*2; k, v 2*64*2; act 2*192*2;
    # tagged 32-bit copies of h, h_mid, q, act; 256 B of counters; each slice
    # rounded to 256; plus one parameter block per stage (4 per layer + lm_head)
    base = (256 + 256 + 512 + 256 + 256 + 768) + (512 + 512 + 1024 + 1536) + 256
    extra = n - base
    n4 = q4.q4_decode_workspace_bytes(q4.LayerTable([layer] * 4, lin(100, 64), hidden=64, M=2))
    extra4 = n4 - base
    assert extra % 256 == 0 and extra4 % 256 == 0
    assert 9 * 128 <= extra <= 9 * 1024 + 255      # 9 stages
    assert 17 * 128 <= extra4 <= 17 * 1024 + 255   # 17 stages
    assert extra4 > extra
    bad = dict(layer, o=lin(64, 96))
    t2 = q4.LayerTable([layer, bad], lin(100, 64), hidden=64, M=2)
    assert L.q4_decode_workspace_bytes(ctypes.byref(t2.t)) == 0
    assert b"layer 1 o" in L.q4_last_error()
    t3 = q4.LayerTable([layer], lin(100, 64), hidden=64, M=9)
    assert L.q4_decode_workspace_bytes(ctypes.byref(t3.t)) == 0
    # A step without a workspace fails on the host.
    assert L.q4_decode_step(ctypes.byref(t.t), FAKE, FAKE, None) == -1


def test_gemm_and_prefill_validation(L):
    d = q4.q4_gemm_desc()
    assert L.q4_gemm(None, None) == -1
    d.M, d.X, d.Y = 4, FAKE, FAKE
    d.w = q4.q4_linear(FAKE, FAKE, FAKE, 128, 64)
    d.mode, d.out_dtype = q4.Q4_GEMV_GLU, q4.Q4_F16
    assert L.q4_gemm(ctypes.byref(d), None) == -1          # GLU without the up matrix
    d.up = q4.q4_linear(FAKE, FAKE, FAKE, 256, 64)
    assert L.q4_gemm(ctypes.byref(d), None) == -1          # gate and up differ
    layer = {"q": lin(128, 64), "k": lin(128, 64), "v": lin(128, 64), "o": lin(64, 128), "gate": lin(256, 64),
             "up": lin(256, 64), "down": lin(64, 256)}
    t = q4.LayerTable([layer], lin(100, 64), hidden=64, M=1)
    n8 = q4.q4_prefill_workspace_bytes(t, 8)
    # n [8][64], q [8][128], k, v [8][128], act [8][256] fp16, each slice rounded
    # to 256 B, then the fp32 partials of split GEMMs: none here (K <= 256 is
    # at most 4 K steps), so one 256-byte slice
    assert n8 == 1024 + 2048 + 2048 + 2048 + 4096 + 256
    assert L.q4_gemm_workspace_bytes(512, 1024, 3072, 0) == 4 * 512 * 1024 * 4   # 32 tiles -> 4 parts of 12 K steps
    assert L.q4_gemm_workspace_bytes(512, 1024, 2048, 1) == 4 * 2 * 512 * 1024 * 4   # 32 tiles -> 4 parts of 8 K steps
    assert L.q4_gemm_workspace_bytes(512, 3072, 1024, 1) == 0                     # 16 K steps: faster unsplit
    assert L.q4_gemm_workspace_bytes(2048, 2048, 1024, 0) == 0                    # 256 tiles: no split
    assert L.q4_gemm_workspace_bytes(512, 1024, 192, 0) == 0                      # 3 K steps: too few to split
    assert L.q4_prefill_workspace_bytes(ctypes.byref(t.t), 0) == 0
    assert L.q4_prefill(ctypes.byref(t.t), FAKE, 4, 0, None, FAKE, n8, None) == -1      # chunk 0
    assert L.q4_prefill(ctypes.byref(t.t), FAKE, 4, 16, None, FAKE * 256, n8, None) == -1  # workspace too small
    assert L.q4_prefill(ctypes.byref(t.t), FAKE, -1, 8, None, FAKE * 256, n8, None) == -1


def test_moe_validation(L):
    assert L.q4_moe_route_workspace_bytes(2048, 128, 8) == 64 * 128 * 4
    args = [FAKE] * 7
    assert L.q4_moe_route(FAKE, 16, 128, 9, *args[:6], FAKE, 1 << 20, None) == -1   # topk > 8
    assert L.q4_moe_route(FAKE, 16, 300, 8, *args[:6], FAKE, 1 << 20, None) == -1   # E > 256
    assert L.q4_moe_route(FAKE, 16, 128, 8, *args[:6], FAKE, 0, None) == -1         # workspace too small
    # token counts whose indices would leave int: refused before anything is enqueued
    assert L.q4_moe_route(FAKE, (1 << 24) + 1, 128, 4, *args[:6], FAKE, 1 << 40, None) == -2
    assert L.q4_moe_route(FAKE, 2**31 - 1, 128, 1, *args[:6], FAKE, 1 << 40, None) == -2
    assert L.q4_moe_gather(FAKE, 4, 12, FAKE, 8, FAKE, None) == -1
    assert L.q4_moe_gather(FAKE + 8, 4, 64, FAKE, 8, FAKE, None) == -3
    assert L.q4_moe_combine(FAKE, 0, 64, FAKE, FAKE, 4, 9, FAKE, 0, None) == -1


def test_attention_validation(L):
    # the (cos, sin) table, (max, sum) per head and 64-position chunk, then the partial outputs
    assert L.q4_attention_workspace_bytes(16, 128, 4096) == 64 * 8 + 16 * 64 * 2 * 4 + 16 * 64 * 128 * 4
    assert L.q4_attention_workspace_bytes(0, 128, 4096) == 0
    assert L.q4_attention(None, None) == -1
    d = q4.q4_attention_desc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 8, 128, 4096, 1e6, FAKE, FAKE * 256, 1 << 20)
    bad = [("head_dim", 96, -2), ("n_kv_heads", 5, -1), ("n_kv_heads", 1, -2), ("rope_theta", 1.0, -1),
           ("workspace_bytes", 100, -1), ("max_seq", 0, -1)]
    for f, v, want in bad:
        e = q4.q4_attention_desc.from_buffer_copy(d)
        setattr(e, f, v)
        assert L.q4_attention(ctypes.byref(e), None) == want, f
    e = q4.q4_attention_desc.from_buffer_copy(d)
    e.k_cache = FAKE + 8
    assert L.q4_attention(ctypes.byref(e), None) == -3


def test_decode_attention_table_validation(L):
    layer = {"q": lin(128, 64), "k": lin(64, 64), "v": lin(64, 64), "o": lin(64, 128), "gate": lin(192, 64),
             "up": lin(192, 64), "down": lin(64, 192), "k_cache": FAKE, "v_cache": FAKE}
    t = q4.LayerTable([layer], lin(100, 64), hidden=64, M=1, flags=q4.Q4_DECODE_ATTENTION, head_dim=64,
                      max_seq=32, pos=FAKE)
    n = L.q4_decode_workspace_bytes(ctypes.byref(t.t))
    plain = q4.q4_decode_workspace_bytes(q4.LayerTable([layer], lin(100, 64), hidden=64, M=1))
    assert n > plain                                   # + the attention output and its scratch
    # the clustered step's tables and exchange region, for tables that ask for it
    assert q4.q4_decode_workspace_bytes(q4.LayerTable([layer], lin(100, 64), hidden=64, M=1,
                                                      flags=q4.Q4_DECODE_CLUSTERED)) > plain
    for kw, frag in ((dict(M=2), b"M = 1"), (dict(head_dim=96), b"head"), (dict(pos=None), b"pos"),
                     (dict(flags=q4.Q4_DECODE_ATTENTION | q4.Q4_DECODE_TAGGED), b"TAGGED")):
        args = dict(hidden=64, M=1, flags=q4.Q4_DECODE_ATTENTION, head_dim=64, max_seq=32, pos=FAKE)
        args.update(kw)
        tb = q4.LayerTable([layer], lin(100, 64), **args)
        assert L.q4_decode_workspace_bytes(ctypes.byref(tb.t)) == 0, kw
        assert frag in L.q4_last_error(), (kw, L.q4_last_error())


def test_binding_refuses_host_tensors(L):
    # a host address handed to a kernel would be dereferenced on the device:
    # the binding refuses a tensor that is not in CUDA memory before any call
    torch = pytest.importorskip("torch")
    host = torch.zeros(64, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA device memory"):
        q4.q4_gemv(host, host, host, host, host, 1, 8, 64)
    with pytest.raises(ValueError, match="CUDA device memory"):
        q4.LayerTable([], (host, host, host, 8, 64), hidden=64, M=1)
