"""Failure detection on the GPU without a fault: the library's bounded waits
(a tagged word nobody writes, an mbarrier nobody arrives on) run out, latch
Q4_ERR_TIMEOUT for the host to read, and leave the context usable."""
import time

import numpy as np
import pytest

import oracle
import q4synth
from helpers import assert_parity, dev_q4, torch_dev

torch = pytest.importorskip("torch")
import bit_quantized_gemv_q4_gb300 as q4  # noqa: E402

pytestmark = pytest.mark.gpu

Q4_ERR_TIMEOUT = -5


def test_expired_waits_are_reported_and_the_context_survives():
    assert q4.q4_device_status() == 0
    t0 = time.time()
    q4.q4_selftest_expired_wait()
    assert q4.q4_device_status() == Q4_ERR_TIMEOUT
    elapsed = time.time() - t0
    assert 3.5 < elapsed < 30.0, elapsed          # two waits of ~2 s each, then the kernel ended
    assert q4.q4_device_status() == 0             # read once, then cleared
    # the context still runs the hot path correctly
    m = q4synth.q4_matrix(31, 256, 1024)
    x = q4synth.activations(32, 1, 1024)
    Wq, s, b = dev_q4(m)
    y = torch.empty(1, 256, device="cuda")
    q4.q4_gemv(Wq, s, b, torch_dev(x), y, 1, 256, 1024)
    assert q4.q4_device_status() == 0
    y_ref, A = oracle.gemv(m.Wq, m.scales, m.biases, x)
    assert_parity(y.cpu().numpy(), y_ref, A)
