"""The allocation-free routing entry point, q4_moe_route_noalloc.

It exists for callers that cannot allocate device memory (a plugin inside a
host runtime that owns every device buffer, a serving loop whose allocations
are fixed at load time): instead of a caller workspace it uses a static
array inside the library.  These tests check, through the C ABI, that it
returns exactly what q4_moe_route returns, on two calls in a row with
different inputs (the shared array keeps the first call's contents), and
that requests beyond the array's size are refused before anything runs.

The file name makes pytest collect it last."""
import ctypes

import numpy as np
import pytest

import q4synth

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from bit_quantized_gemv_q4_gb300 import build
    build.build()


def route_both(T, E, k, seed):
    logits = torch.from_numpy(q4synth.router_logits(seed, T, E)).cuda()
    R = T * k

    def bufs():
        return dict(ids=torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
                    w=torch.full((T, k), float("nan"), device="cuda"),
                    off=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
                    tok=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                    eid=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                    pos=torch.full((T, k), -7, dtype=torch.int32, device="cuda"))

    a, b = bufs(), bufs()
    nws = q4.q4_moe_route_workspace_bytes(T, E, k)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    q4.q4_moe_route(logits, T, E, k, a["ids"], a["w"], a["off"], a["tok"], a["eid"], a["pos"], ws, nws)
    q4.q4_moe_route_noalloc(logits, T, E, k, b["ids"], b["w"], b["off"], b["tok"], b["eid"], b["pos"])
    torch.cuda.synchronize()
    assert q4.q4_device_status() == 0
    return {n: v.cpu().numpy() for n, v in a.items()}, {n: v.cpu().numpy() for n, v in b.items()}


@pytest.mark.gpu
def test_noalloc_route_matches_workspace_route_twice():
    # calls in a row; the second uses more blocks than the first, so it
    # cannot pass on counters left over from the first; then the exact fit
    # (ceil(T/32) * E = 65536 counters) and a ragged last block (T % 32 != 0)
    for T, seed in ((512, 501), (2048, 502), (16384, 503), (1000, 504)):
        ref, got = route_both(T, 128, 8, seed)
        for n in ("ids", "off", "tok", "eid", "pos"):
            assert np.array_equal(ref[n], got[n]), (T, n)
        assert np.max(np.abs(ref["w"] - got["w"])) <= 1e-6


def test_noalloc_rejects_requests_beyond_the_static_scratch():
    L = q4.lib()
    fake = 0x10000
    # 16384 tokens x 128 experts fit (512 blocks x 128 = 65536 counters); one more block does not
    st = L.q4_moe_route_noalloc(fake, 16384 + 32, 128, 8, *([fake] * 6), None)
    assert st == -2
    assert b"static scratch" in L.q4_last_error()
    st = L.q4_moe_route_noalloc(fake, 16, 128, 9, *([fake] * 6), None)
    assert st == -1
    # the block count is formed without int overflow: the largest int is refused
    st = L.q4_moe_route_noalloc(fake, 2**31 - 1, 128, 8, *([fake] * 6), None)
    assert st == -2
