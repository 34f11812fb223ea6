"""Per-phase latency breakdown of the clustered decode step (a diagnostic).

Builds a separate copy of the library with the step kernel's timestamp
points compiled in (-DQ4_STEP_TRACE, into _build_trace/), runs the
Qwen3-0.6B-shaped decode step (M = 1, random Q4 weights drawn on the device)
with Q4_DECODE_CLUSTERED, and prints, for the first and the last CTA of the
grid, the median over layers 2..L-1 of the time between consecutive phase
points of a layer (the consumer warps, the layer's critical path), and the
k / v kernel's points as offsets from the layer's start.  The timestamps come from %globaltimer, so they include
every wait; the per-step time is taken with CUDA events over 200 steps of
the ordinary replay (the trace build writes a few extra global words)."""
from __future__ import annotations

import ctypes
import json
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)

PHASES = ["layer start", "q rows done", "q sent", "q block in", "o partial", "published", "h' collected",
          "h' in", "gate/up rows done", "act sent", "act block in", "down partial", "published", "h collected",
          "h in"]
# the k / v kernel's first CTA (off the critical path), reported as offsets
# from the clustered kernel's layer start
SIDE_POINTS = {20: "k/v kernel: layer's x staged", 21: "k/v kernel: k, v rows stored"}


def build_traced() -> str:
    from bit_quantized_gemv_q4_gb300 import build as b
    obj = os.path.join(HERE, "_build_trace")
    os.makedirs(obj, exist_ok=True)
    lib = os.path.join(obj, "libq4gb300_trace.so")
    srcs = sorted(f for f in os.listdir(b.CSRC) if f.endswith(".cu"))
    procs, objs = [], []
    for f in srcs:
        o = os.path.join(obj, f + ".o")
        procs.append(subprocess.Popen([b.nvcc(), *b.ARCH, *b.FLAGS, "-DQ4_STEP_TRACE", "-c",
                                       os.path.join(b.CSRC, f), "-o", o]))
        objs.append(o)
    if any(p.wait() != 0 for p in procs):
        raise RuntimeError("nvcc failed")
    subprocess.run([b.nvcc(), *b.ARCH, "-shared", "-cudart", "shared", "-o", lib, *objs], check=True)
    return lib


def main():
    import torch

    import bit_quantized_gemv_q4_gb300 as q4
    import q4synth
    q4.LIB_PATH = build_traced()
    L = q4.lib()
    L.q4_step_trace_read.argtypes = [ctypes.c_void_p]
    shape = q4synth.QWEN3_0P6B
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(5)

    def mat(N, K):
        Wq = torch.randint(-2**31, 2**31 - 1, (N, K // 8), dtype=torch.int32, device=dev, generator=gen)
        s = (torch.rand(N, K // 64, device=dev, generator=gen) * 0.005).half()
        return (Wq, s, (-8 * s.float()).half(), N, K)

    dl = [{nm: mat(N, K) for nm, N, K in shape.layer_linears()} for _ in range(shape.n_layers)]
    dlm = mat(shape.vocab, shape.hidden)
    t = q4.LayerTable(dl, dlm, hidden=shape.hidden, M=1, flags=q4.Q4_DECODE_CLUSTERED)
    nws = q4.q4_decode_workspace_bytes(t)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    t.set_workspace(ws, nws)
    x = torch.from_numpy(q4synth.activations(1, 1, shape.hidden)).to(dev)
    lg = torch.empty(1, shape.vocab, device=dev)
    for _ in range(30):
        q4.q4_decode_step(t, x, lg)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(200):
        q4.q4_decode_step(t, x, lg)
    e1.record()
    torch.cuda.synchronize()
    buf = np.zeros(2 * 4096, dtype=np.uint64)
    if L.q4_step_trace_read(buf.ctypes.data) != 0:
        raise RuntimeError("trace read failed")
    out = {"shape": shape.name, "path": q4.q4_decode_path(t), "ms_per_step": e0.elapsed_time(e1) / 200,
           "device_status": q4.q4_device_status()}
    nl = shape.n_layers
    for cta, name in ((0, "first CTA"), (1, "last CTA")):
        tr = buf[cta * 4096: cta * 4096 + nl * 32].reshape(nl, 32).astype(np.int64)
        lay = [int(tr[l + 1, 0] - tr[l, 0]) for l in range(nl - 1)]
        phases = {}
        for a in range(len(PHASES) - 1):
            d = [int(tr[l, a + 1] - tr[l, a]) for l in range(2, nl - 1)]
            phases[f"{PHASES[a]} -> {PHASES[a + 1]}"] = int(np.median(d))
        side = {nm: int(np.median([tr[l, k] - tr[l, 0] for l in range(2, nl - 1)])) for k, nm in SIDE_POINTS.items()}
        out[name] = {"layer_ns_median": int(np.median(lay)), "phase_ns_median": phases,
                     "off_path_ns_after_layer_start": side}
    print(json.dumps(out, indent=1))
    t.release()


if __name__ == "__main__":
    main()
