"""Shared test helpers: moving seeded inputs to the device and the parity bar.

Parity bar (per output element, against the fp64 oracle):
  * fp32 outputs:  |y - y_ref| <= 1e-3 * A    with A = sum_k |w_k x_k|,
                   and ||y - y_ref||_2 / ||y_ref||_2 <= 1e-3;
  * fp16 outputs:  |y - y_ref| <= 1e-3 * A + ulp16(y_ref)  (the fp16 store may
                   round either way of a value within the fp32 error), and the
                   same relative L2 bound.
A = 0 forces an exact 0."""
from __future__ import annotations

import numpy as np

REL_L2 = 1e-3
ELEM = 1e-3


def torch_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def dev_q4(m):
    """Device copies of a q4synth.Q4Matrix (Wq as int32 view of the words)."""
    return torch_dev(m.Wq), torch_dev(m.scales), torch_dev(m.biases)


def ulp16(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def parity_report(y, y_ref, A, fp16_out=False):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = ELEM * A + (ulp16(y_ref) if fp16_out else 0.0)
    bad = err > bound
    nref = np.linalg.norm(y_ref)
    rel = float(np.linalg.norm(y - y_ref) / nref) if nref > 0 else float(np.linalg.norm(y - y_ref))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(A > 0, err / np.where(A > 0, A, 1), np.where(err > 0, np.inf, 0))
    return {"n_bad": int(bad.sum()), "rel_l2": rel, "max_err_over_A": float(ratio.max()) if ratio.size else 0.0,
            "first_bad": np.argwhere(bad)[:5].tolist()}


def assert_parity(y, y_ref, A, fp16_out=False, what=""):
    r = parity_report(y, y_ref, A, fp16_out)
    assert r["n_bad"] == 0, f"{what}: {r}"
    assert r["rel_l2"] <= REL_L2, f"{what}: {r}"
    return r
