"""Benchmark: Q4 decode-step matmul stream on one GB300 (or N replicas).

Workload: the Qwen3-0.6B-shaped decode weight stream at M = 1 -- 28 layers of
fused QKV (1024 -> 2048+1024+1024), o (2048 -> 1024, + residual), fused
gate/up (1024 -> 2x3072, SiLU*up), down (3072 -> 1024, + residual), then
lm_head (1024 -> 151936); Q4 group-64 weights with fp16 scale and bias,
synthetic and seeded (random-init of that shape; no trained weights).  One
step = one decode token = one replay of the captured stream: by default the
clustered step (Q4_DECODE_CLUSTERED: the layer stack as one launch of
thread-block clusters, the k / v rows beside it, then lm_head: 3 kernels),
with `--decode-path per-stage` the 113 GEMV launches.

Prints ONE JSON line (rank 0).  `value` is whole-job decode tok/s with the
inputs resident in HBM; `e2e` is the same through the C ABI with the input
vector copied in from pinned host memory and the logits copied out every step;
`roofline` is the step's kernels against the measured HBM copy bandwidth
(algorithmic bytes per step / step time; the per-kernel shares are in the
committed ncu launch list); `cpu_baseline` is the fp64 CPU
oracle timed on the host cores on a bounded sample.  `--impl reference` times
the oracle instead (the reference arm).

Multi-GPU: replicas only (the path does not shard); each rank decodes its own
stream, value = ranks x tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4 fused-dequant GEMV HBM GB/s (% of peak); decode-step matmul tok/s"
FALLBACK_HBM_GBS = 6800.0


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (context beside the measured copy bandwidth)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(path: str = "per-stage") -> str:
    """Hash of the decode kernels' code (q4_gemv.cu + q4_device.cuh, and
    q4_step.cu for the clustered step) with comments and whitespace removed:
    a comment edit keeps the recorded ncu traffic valid, any code change in
    those files invalidates it (the traffic is then re-captured)."""
    h = hashlib.sha256()
    for nm in (("q4_gemv.cu", "q4_device.cuh") + (("q4_step.cu",) if path == "clustered" else ())):
        with open(os.path.join(ROOT, "bit_quantized_gemv_q4_gb300", "csrc", nm), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", " ", src)                   # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


TRAFFIC_FILES = {"per-stage": "q4_gemv_decode_qwen3_0p6b_traffic.txt",
                 "clustered": "q4_step_decode_qwen3_0p6b_traffic.txt"}


def recorded_traffic(path: str = "per-stage"):
    """DRAM bytes per step and launches per step of the decode path from the
    committed ncu summary, or None if it was taken with a different kernel
    source."""
    fn = os.path.join(ROOT, "profiles", TRAFFIC_FILES[path])
    try:
        kv = {}
        for ln in open(fn):
            if "=" in ln and not ln.startswith("#"):
                k, v = ln.split("=", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_hash") != kernel_source_hash(path):
            return None
        return float(kv["dram_bytes_per_step"]), int(kv["launches_per_step"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 5.0  # the first reading, so sampling covers the region
            while not self.lines and time.time() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        time.sleep(0.25)  # let the reading that follows the region arrive

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        """Median SM clock and active slowdown reasons over the readings taken
        inside [start, stop]; a region shorter than the 100 ms reading period
        uses the first reading after it (noted in "window")."""
        t0 = self.t0 if self.t0 is not None else 0.0
        t1 = self.t1 if self.t1 is not None else float("inf")
        inside = [ln for ts, ln in self.lines if t0 <= ts <= t1]
        window = "timed region"
        if not inside:
            after = [ln for ts, ln in self.lines if ts > t1][:1]
            inside, window = after, "first reading after the timed region (region shorter than 100 ms)"
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
            p = [v.strip() for v in ln.split(",")]
            if len(p) < 7:
                continue
            try:
                sm.append(float(p[0]))
                mx = max(mx, float(p[1]))
            except ValueError:
                continue
            for nm, v in zip(names, p[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "window": window}


# ------------------------------------------------------------------ workload

def make_model(shape, device, layers=True):
    import torch

    import q4synth

    def dev(m):
        return (torch.from_numpy(m.Wq.view("int32")).to(device), torch.from_numpy(m.scales).to(device),
                torch.from_numpy(m.biases).to(device), m.N, m.K)

    if not layers:  # the lm_head alone, with the seed the whole stack gives it
        lm = q4synth.q4_matrix(q4synth.BASE_SEED + 16 * shape.n_layers, shape.vocab, shape.hidden)
        return None, dev(lm), None
    layers, lm = q4synth.decode_weights(shape)
    return [{k: dev(v) for k, v in d.items()} for d in layers], dev(lm), (layers, lm)


def cpu_oracle_rate(shape, host_model, seconds: float, one_sample: bool = False, nthreads: int = 0):
    """Oracle throughput on a bounded sample, as decode tok/s of the full step.

    Sample i = layer (i mod L)'s seven matrices plus the (i mod L)-th of L
    equal slices of lm_head rows: together 1/L of a step's weights.
    nthreads 0 = the oracle's OpenMP default (all cores)."""
    import numpy as np

    import oracle
    import q4synth
    layers, lm = host_model
    L = shape.n_layers
    x = q4synth.activations(q4synth.BASE_SEED + 4242, 1, shape.hidden)
    xs = {}
    done_w, t_total, i = 0, 0.0, 0
    while True:
        li = i % L
        t0 = time.perf_counter()
        w = 0
        for nm, N, K in shape.layer_linears():
            m = layers[li][nm]
            if K not in xs:
                xs[K] = q4synth.activations(q4synth.BASE_SEED + 4243 + K, 1, K)
            oracle.gemv(m.Wq, m.scales, m.biases, xs[K], nthreads=nthreads)
            w += N * K
        rows = np.arange(li * shape.vocab // L, (li + 1) * shape.vocab // L)
        oracle.gemv(lm.Wq, lm.scales, lm.biases, x, rows=rows, nthreads=nthreads)
        w += rows.size * shape.hidden
        t_total += time.perf_counter() - t0
        done_w += w
        i += 1
        if one_sample or t_total >= seconds:
            break
    return done_w / t_total / shape.weights_per_step(), i, t_total


def moe_prefill(device, iters: int = 20, warmup: int = 5, token_counts=(128, 512, 2048)):
    """MoE prefill layer (Qwen3-30B-A3B-shaped: 128 experts, top-8, hidden
    2048, expert FFN 768): route -> gather -> gate/up GEMM (SiLU*up) -> down
    GEMM -> combine, timed with CUDA events per stage and as a whole."""
    import torch

    import bit_quantized_gemv_q4_gb300 as q4
    import q4synth
    S = q4synth.QWEN3_30B_A3B_MOE
    E, k, H, F = S.experts, S.topk, S.hidden, S.ffn
    gu, dn = q4synth.moe_weights(S)

    def dev(m):
        return (torch.from_numpy(m.Wq.view("int32")).to(device), torch.from_numpy(m.scales).to(device),
                torch.from_numpy(m.biases).to(device))

    dgu, ddn = dev(gu), dev(dn)
    weight_bytes = gu.nbytes() + dn.nbytes()
    stream = torch.cuda.current_stream(device)
    out = {"shape": f"{S.name}: E={E} top{k} hidden={H} ffn={F}", "weight_bytes": weight_bytes}
    for T in token_counts:
        R = T * k
        logits = torch.from_numpy(q4synth.router_logits(q4synth.BASE_SEED + 7 + T, T, E)).to(device)
        X = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 8 + T, T, H)).to(device)
        ids = torch.empty(T, k, dtype=torch.int32, device=device)
        w = torch.empty(T, k, device=device)
        off = torch.empty(E + 1, dtype=torch.int32, device=device)
        tok = torch.empty(R, dtype=torch.int32, device=device)
        eid = torch.empty(R, dtype=torch.int32, device=device)
        pos = torch.empty(T, k, dtype=torch.int32, device=device)
        nws = q4.q4_moe_route_workspace_bytes(T, E, k)
        ws = torch.empty(nws, dtype=torch.uint8, device=device)
        Xs = torch.empty(R, H, dtype=torch.float16, device=device)
        Hh = torch.empty(R, F, dtype=torch.float16, device=device)
        Y = torch.empty(R, H, dtype=torch.float16, device=device)
        o = torch.empty(T, H, dtype=torch.float16, device=device)
        def layer(ev=None):
            if ev:
                ev[0].record(stream)
            q4.q4_moe_route(logits, T, E, k, ids, w, off, tok, eid, pos, ws, nws, stream)
            q4.q4_moe_gather(X, T, H, tok, R, Xs, stream)
            if ev:
                ev[1].record(stream)
            q4.q4_moe_gemm(*dgu, Xs, eid, off, Hh, E, F, H, R, q4.Q4_GEMV_GLU, q4.Q4_F16, stream)
            if ev:
                ev[2].record(stream)
            q4.q4_moe_gemm(*ddn, Hh, eid, off, Y, E, H, F, R, q4.Q4_GEMV_PLAIN, q4.Q4_F16, stream)
            if ev:
                ev[3].record(stream)
            q4.q4_moe_combine(Y, q4.Q4_F16, H, pos, w, T, k, o, q4.Q4_F16, stream)
            if ev:
                ev[4].record(stream)

        for _ in range(warmup):
            layer()
        torch.cuda.synchronize(device)
        # Enqueue every timed layer, synchronise once: the host runs ahead of
        # the GPU, so the events measure device time, not launch gaps.
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(iters)]
        for i in range(iters):
            layer(evs[i])
        torch.cuda.synchronize(device)
        tot = {"route_gather": 0.0, "gate_up": 0.0, "down": 0.0, "combine": 0.0}
        for ev in evs:
            tot["route_gather"] += ev[0].elapsed_time(ev[1])
            tot["gate_up"] += ev[1].elapsed_time(ev[2])
            tot["down"] += ev[2].elapsed_time(ev[3])
            tot["combine"] += ev[3].elapsed_time(ev[4])
        if q4.q4_device_status(stream) != 0:
            raise RuntimeError("device status after MoE timing")
        us = {kk: 1000 * v / iters for kk, v in tot.items()}
        gemm_us = us["gate_up"] + us["down"]
        flops = 2.0 * R * (2 * F * H + H * F)
        out[f"T={T}"] = {
            "layer_us": sum(us.values()), **{f"{kk}_us": v for kk, v in us.items()},
            "gemm_tflops": flops / (gemm_us * 1e-6) / 1e12,
            "gemm_weight_gbs": weight_bytes / (gemm_us * 1e-6) / 1e9,
            "prefill_tok_per_s": T / (sum(us.values()) * 1e-6),
        }
    return out


def tensor_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s, burst); fp16 runs at the same rate."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 same rate)"
    except Exception:
        return 1900.0, "fallback"


def dense_prefill(device, dl, dlm, shape, iters: int = 5, warmup: int = 3, cases=((512, 512), (2048, 512),
                                                                                  (2048, 2048))):
    """Chunked prefill of the whole layer stack (q4_prefill: per chunk and
    layer an RMSNorm kernel and five tensor-core GEMMs, then the lm_head GEMV
    of the last token), as (prompt tokens, chunk) cases; the prompt is reset
    from a resident copy before each timed call (a device copy inside the
    timed region, <1 % of it)."""
    import torch

    import bit_quantized_gemv_q4_gb300 as q4
    import q4synth
    table = q4.LayerTable(dl, dlm, hidden=shape.hidden, M=1)
    stream = torch.cuda.current_stream(device)
    per_tok = 2.0 * sum(N * K for _, N, K in shape.layer_linears()) * shape.n_layers
    peak, kind = tensor_peak()
    out = {"shape": f"{shape.name}, {shape.n_layers} layers", "peak_tflops": peak, "peak_kind": kind}
    for T, C in cases:
        x0 = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 9100 + T, T, shape.hidden)).to(device)
        h = torch.empty_like(x0)
        nws = q4.q4_prefill_workspace_bytes(table, C)
        ws = torch.empty(nws, dtype=torch.uint8, device=device)
        lg = torch.empty(shape.vocab, dtype=torch.float32, device=device)
        for _ in range(warmup):
            h.copy_(x0)
            q4.q4_prefill(table, h, T, C, lg, ws, nws, stream)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            h.copy_(x0)
            q4.q4_prefill(table, h, T, C, lg, ws, nws, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        if q4.q4_device_status(stream) != 0:
            raise RuntimeError("device status after prefill timing")
        ms = e0.elapsed_time(e1) / iters
        tf = per_tok * T / (ms * 1e-3) / 1e12
        out[f"T={T} chunk={C}"] = {"ms": ms, "tok_per_s": T / (ms * 1e-3), "gemm_tflops": tf,
                                   "tensor_frac": tf / peak}
    table.release()
    # with attention (the prompt fills a KV cache; head_dim 128: 16 q / 8 kv heads)
    hd = 128
    hkv = shape.kv // hd
    T, C = 2048, 2048
    caches = [(torch.zeros(hkv, T, hd, dtype=torch.float16, device=device),
               torch.zeros(hkv, T, hd, dtype=torch.float16, device=device)) for _ in range(shape.n_layers)]
    pos = torch.zeros(1, dtype=torch.int32, device=device)
    ta = q4.LayerTable([dict(d, k_cache=kc, v_cache=vc) for d, (kc, vc) in zip(dl, caches)], dlm,
                       hidden=shape.hidden, M=1, flags=q4.Q4_DECODE_ATTENTION, head_dim=hd, max_seq=T, pos=pos)
    x0 = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 9200, T, shape.hidden)).to(device)
    h = torch.empty_like(x0)
    nws = q4.q4_prefill_workspace_bytes(ta, C)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    lg = torch.empty(shape.vocab, dtype=torch.float32, device=device)
    times = []
    for it in range(warmup + iters):
        h.copy_(x0)
        pos.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q4.q4_prefill(ta, h, T, C, lg, ws, nws, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        if it >= warmup:
            times.append(e0.elapsed_time(e1))
    if q4.q4_device_status(stream) != 0:
        raise RuntimeError("device status after prefill-with-attention timing")
    ms = sum(times) / len(times)
    out[f"T={T} chunk={C} attention"] = {"ms": ms, "tok_per_s": T / (ms * 1e-3)}
    ta.release()
    return out


def decode_attention(device, dl, dlm, shape, contexts=(1024, 4096), steps: int = 200, warmup: int = 10):
    """Decode step with attention (Q4_DECODE_ATTENTION, M = 1): the weight
    stream plus RoPE, KV-cache append and attention over `context` cached
    positions (random fp16 cache contents; head_dim 128, so 16 query and 8
    kv heads on the Qwen3-0.6B shape).  Graph replays back to back."""
    import torch

    import bit_quantized_gemv_q4_gb300 as q4
    import q4synth
    hd = 128
    hkv = shape.kv // hd
    out = {"shape": f"{shape.name}, head_dim {hd}, {shape.q // hd} q / {hkv} kv heads"}
    max_seq = max(contexts) + steps + warmup + 1
    gen = torch.Generator(device=device).manual_seed(77)
    caches = [(torch.randn(hkv, max_seq, hd, device=device, generator=gen).half(),
               torch.randn(hkv, max_seq, hd, device=device, generator=gen).half()) for _ in range(shape.n_layers)]
    layers = [dict(d, k_cache=kc, v_cache=vc) for d, (kc, vc) in zip(dl, caches)]
    pos = torch.zeros(1, dtype=torch.int32, device=device)
    table = q4.LayerTable(layers, dlm, hidden=shape.hidden, M=1, flags=q4.Q4_DECODE_ATTENTION, head_dim=hd,
                          max_seq=max_seq, pos=pos)
    nws = q4.q4_decode_workspace_bytes(table)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    table.set_workspace(ws, nws)
    x = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4244, 1, shape.hidden)).to(device)
    logits = torch.empty(1, shape.vocab, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for ctx in contexts:
        pos.fill_(ctx)
        for _ in range(warmup):
            q4.q4_decode_step(table, x, logits, stream)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            q4.q4_decode_step(table, x, logits, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        if q4.q4_device_status(stream) != 0:
            raise RuntimeError("device status after attention timing")
        ms = e0.elapsed_time(e1) / steps
        n_mid = ctx + warmup + steps / 2
        kv_bytes = shape.n_layers * 2 * hkv * n_mid * hd * 2
        byts = shape.weight_bytes_per_step() + kv_bytes
        out[f"context={ctx}"] = {"ms": ms, "tok_per_s": 1000.0 / ms, "kv_bytes_per_step": kv_bytes,
                                 "gbs": byts / (ms * 1e-3) / 1e9}
    table.release()
    return out


def q8_lm_head(q4, device, M: int = 1):
    """The lm_head-shaped GEMV (N=151936, K=1024) with 8-bit codes: 8 warm-up
    launches, then 64 timed over 4 distinct weight copies (4 x 166 MB > L2)."""
    import torch

    import q4synth
    N, K = 151936, 1024
    mats = []
    for i in range(4):
        g = torch.Generator(device=device).manual_seed(200 + i)
        Wq = torch.randint(-2**31, 2**31 - 1, (N, K // 4), dtype=torch.int32, device=device, generator=g)
        s = (torch.rand(N, K // 64, device=device, generator=g) * 2e-4).half()
        mats.append((Wq, s, (-128 * s.float()).half()))
    x = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4243, M, K)).to(device)
    y = torch.empty(M, N, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for i in range(8):
        q4.q4_gemv8(*mats[i % 4], x, y, M, N, K, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(64):
        q4.q4_gemv8(*mats[i % 4], x, y, M, N, K, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / 64
    nb = N * K * (1.0 + 4.0 / 64) + K * 2 * M + N * 4 * M
    peak, kind = peaks()
    return {"ms": ms, "gbs": nb / (ms / 1000.0) / 1e9, "frac": nb / (ms / 1000.0) / 1e9 / peak, "peak_kind": kind,
            "shape": f"M={M} N={N} K={K}, 8-bit codes (1.0625 B/weight), 4 rotating copies"}


def decode_streams(device, steps: int = 200, warmup: int = 10):
    """Decode steps of the larger stacks the parity tests cover: Llama-3.2-3B
    shaped at M = 1 and M = 4, Qwen3-4B shaped at M = 1 (random Q4 weights
    drawn on the device; 1.8-2.3 GB per step, so no L2 reuse); at M = 1 also
    with the clustered step (Q4_DECODE_CLUSTERED)."""
    import torch

    import bit_quantized_gemv_q4_gb300 as q4
    import q4synth
    peak, kind = peaks()
    out = {"peak_kind": kind}
    for shape, M in ((q4synth.LLAMA32_3B, 1), (q4synth.LLAMA32_3B, 4), (q4synth.QWEN3_4B, 1)):
        gen = torch.Generator(device=device).manual_seed(4000 + M)

        def mat(N, K):
            Wq = torch.randint(-2**31, 2**31 - 1, (N, K // 8), dtype=torch.int32, device=device, generator=gen)
            s = (torch.rand(N, K // 64, device=device, generator=gen) * 0.005).half()
            return (Wq, s, (-8 * s.float()).half(), N, K)

        dl = [{nm: mat(N, K) for nm, N, K in shape.layer_linears()} for _ in range(shape.n_layers)]
        dlm = mat(shape.vocab, shape.hidden)
        for flags in ((0, q4.Q4_DECODE_CLUSTERED) if M == 1 else (0,)):
            table = q4.LayerTable(dl, dlm, hidden=shape.hidden, M=M, flags=flags)
            nws = q4.q4_decode_workspace_bytes(table)
            ws = torch.empty(nws, dtype=torch.uint8, device=device)
            table.set_workspace(ws, nws)
            x = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4246, M, shape.hidden)).to(device)
            logits = torch.empty(M, shape.vocab, dtype=torch.float32, device=device)
            stream = torch.cuda.current_stream(device)
            for _ in range(warmup):
                q4.q4_decode_step(table, x, logits, stream)
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                q4.q4_decode_step(table, x, logits, stream)
            e1.record(stream)
            torch.cuda.synchronize(device)
            if q4.q4_device_status(stream) != 0:
                raise RuntimeError("device status after stream timing")
            ms = e0.elapsed_time(e1) / steps
            gbs = shape.weight_bytes_per_step() / (ms * 1e-3) / 1e9  # weight bytes only (activations < 0.1 %)
            key = f"{shape.name} M={M}" + (" clustered" if flags else "")
            out[key] = {"ms": ms, "tok_per_s": M * 1000.0 / ms, "path": q4.q4_decode_path(table),
                        "launches": 2 if q4.q4_decode_path(table) == 3 else 4 * shape.n_layers + 1,
                        "weight_bytes": shape.weight_bytes_per_step(), "gbs": gbs, "frac": gbs / peak}
            table.release()
            del table, ws
        del dl, dlm
        torch.cuda.empty_cache()
    return out


def bits_lm_head(q4, device, widths=(2, 3, 5, 6)):
    """The lm_head-shaped GEMV (M=1, N=151936, K=1024) with b-bit codes:
    8 warm-up launches, then 64 timed over 4 distinct weight copies (> L2)."""
    import torch

    import q4synth
    N, K = 151936, 1024
    peak, kind = peaks()
    x = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4245, 1, K)).to(device)
    y = torch.empty(1, N, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    out = {}
    for bits in widths:
        mats = []
        for i in range(4):
            g = torch.Generator(device=device).manual_seed(300 + 10 * bits + i)
            Wq = torch.randint(-2**31, 2**31 - 1, (N, K * bits // 32), dtype=torch.int32, device=device, generator=g)
            s = (torch.rand(N, K // 64, device=device, generator=g) * 4e-3 / 2 ** bits).half()
            mats.append((Wq, s, (-(2 ** (bits - 1)) * s.float()).half()))
        for i in range(8):
            q4.q4_gemv_bits(*mats[i % 4], x, y, 1, N, K, bits, stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(64):
            q4.q4_gemv_bits(*mats[i % 4], x, y, 1, N, K, bits, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / 64
        nb = N * K * (bits / 8.0 + 4.0 / 64) + K * 2 + N * 4
        out[str(bits)] = {"ms": ms, "gbs": nb / (ms / 1000.0) / 1e9, "frac": nb / (ms / 1000.0) / 1e9 / peak,
                          "bytes_per_weight": bits / 8.0 + 4.0 / 64, "peak_kind": kind}
        del mats
    return out


def decode_clustered(q4, device, dl, dlm, shape, x, steps: int = 1000, warmup: int = 20):
    """The same decode step through the clustered path (Q4_DECODE_CLUSTERED:
    the layer stack as one launch of thread-block clusters with two grid-wide
    hand-offs per layer, the k / v rows as a second launch on the free SMs,
    then lm_head), device-resident, one timed region of `steps` steps."""
    import torch
    table = q4.LayerTable(dl, dlm, hidden=shape.hidden, M=1, flags=q4.Q4_DECODE_CLUSTERED)
    nws = q4.q4_decode_workspace_bytes(table)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    table.set_workspace(ws, nws)
    logits = torch.empty(1, shape.vocab, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        q4.q4_decode_step(table, x, logits, stream)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        q4.q4_decode_step(table, x, logits, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    if q4.q4_device_status(stream) != 0:
        raise RuntimeError("device status after the clustered-step timing")
    ms = e0.elapsed_time(e1) / steps
    path = q4.q4_decode_path(table)
    table.release()
    return {"ms": ms, "tok_per_s": 1000.0 / ms, "path": path, "launches_per_step": 3 if path == 3 else None}


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: replicas run independently, so the job takes
    as long as its slowest replica (all-reduce MAX when world > 1)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, tokens_per_rank_step: int, steps: int, ms_max: float) -> float:
    """Whole-job tokens per second: every rank decodes its own tokens."""
    return world * tokens_per_rank_step * steps / (ms_max / 1000.0)


def decode_per_stage(q4, device, dl, dlm, shape, x, steps: int = 1000, warmup: int = 20):
    """The same 0.6B-shaped step through the per-stage path (113 GEMV
    launches per step, graph + PDL): context beside the clustered headline."""
    import torch
    table = q4.LayerTable(dl, dlm, hidden=shape.hidden, M=1)
    nws = q4.q4_decode_workspace_bytes(table)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    table.set_workspace(ws, nws)
    lg = torch.empty(1, shape.vocab, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        q4.q4_decode_step(table, x, lg, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(steps):
        q4.q4_decode_step(table, x, lg, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    path = q4.q4_decode_path(table)
    if q4.q4_device_status(stream) != 0:
        raise RuntimeError("device status after the per-stage decode timing")
    table.release()
    return {"ms": ms, "tok_per_s": 1000.0 / ms, "path": path, "launches_per_step": 4 * shape.n_layers + 1}


def single_gemv(q4, device, isolated: int = 50, replays: int = 5):
    """The single small GEMV (M = 1, K = 1024, N = 3072, 1.78 MB) three ways:
    isolated (one launch between synchronisations, median of 50 over distinct
    weight copies), and in steady state over a rotating pool of distinct
    copies totalling more than 3x L2 launched back to back from one CUDA
    graph (so no launch hits L2; best and median of 5 replays) -- once with
    programmatic dependent launch (q4_gemv_ex with Q4_GEMV_EARLY_WEIGHTS: each
    launch streams its weights while the one before it finishes; the
    protocol's steady state) and once with plain launches (q4_gemv)."""
    import statistics

    import torch

    import q4synth
    N, K, M = 3072, 1024, 1
    nb = N * K * 0.5625 + K * 2 * M + N * 4 * M
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
    n_copies = int(-(-3 * l2 // int(nb)))
    gen = torch.Generator(device=device).manual_seed(q4synth.BASE_SEED + 8800)
    copies = []
    for _ in range(n_copies):
        Wq = torch.randint(-2**31, 2**31 - 1, (N, K // 8), dtype=torch.int32, device=device, generator=gen)
        sc = (torch.rand(N, K // 64, device=device, generator=gen) * 0.005).half()
        copies.append((Wq, sc, (-8 * sc.float()).half()))
    x = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 8801, M, K)).to(device)
    y = torch.empty(M, N, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for c in copies:  # warm-up: every copy once
        q4.q4_gemv(*c, x, y, M, N, K, stream)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    iso = []
    for i in range(isolated):
        torch.cuda.synchronize(device)
        e0.record(stream)
        q4.q4_gemv(*copies[i % n_copies], x, y, M, N, K, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        iso.append(e0.elapsed_time(e1))
    def steady(early: bool):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in copies:  # the capture stream is current here
                if early:
                    q4.q4_gemv_ex([q4.Segment(*c, N, y=y)], x, M, K, flags=q4.Q4_GEMV_EARLY_WEIGHTS)
                else:
                    q4.q4_gemv(*c, x, y, M, N, K)
        torch.cuda.synchronize(device)
        g.replay()
        torch.cuda.synchronize(device)
        per = []
        for _ in range(replays):
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize(device)
            per.append(e0.elapsed_time(e1) / n_copies)
        del g
        return min(per), statistics.median(per)

    best, med = steady(True)
    best_plain, med_plain = steady(False)
    if q4.q4_device_status(stream) != 0:
        raise RuntimeError("device status after the single-GEMV timing")
    peak, kind = peaks()
    iso_ms = statistics.median(iso)
    gbs = lambda ms: nb / (ms / 1000.0) / 1e9  # noqa: E731
    return {"shape": f"M={M} N={N} K={K}", "bytes_per_launch": nb, "peak_kind": kind,
            "isolated_us": iso_ms * 1000.0, "isolated_gbs": gbs(iso_ms),
            "steady_copies": n_copies, "steady": "graph of back-to-back launches with programmatic dependent "
                                                 "launch (Q4_GEMV_EARLY_WEIGHTS)",
            "steady_us_best": best * 1000.0, "steady_us_median": med * 1000.0,
            "steady_gbs_best": gbs(best), "steady_frac_of_measured": gbs(best) / peak,
            "steady_frac_of_nominal": gbs(best) / NOMINAL_HBM_GBS,
            "plain_launches": {"us_best": best_plain * 1000.0, "us_median": med_plain * 1000.0,
                               "gbs_best": gbs(best_plain), "frac_of_measured": gbs(best_plain) / peak}}


def lm_head_ms(q4, dlm, x, M, stream, device):
    """The largest single launch alone (the lm_head GEMV shape): 8 warm-up
    launches, then 64 timed back to back over 4 distinct weight copies
    (350 MB > L2, so no launch hits in L2)."""
    import torch
    Wq, s, b, N, K = dlm
    mats = [(Wq, s, b)]
    for i in range(3):
        g = torch.Generator(device=device).manual_seed(100 + i)
        mats.append((torch.randint(-2**31, 2**31 - 1, Wq.shape, dtype=torch.int32, device=device, generator=g),
                     s.roll(i + 1, 0).contiguous(), b.roll(i + 1, 0).contiguous()))
    yv = torch.empty(M, N, dtype=torch.float32, device=device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(8):
        q4.q4_gemv(*mats[i % 4], x, yv, M, N, K, stream)
    e0.record(stream)
    for i in range(64):
        q4.q4_gemv(*mats[i % 4], x, yv, M, N, K, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / 64


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)  # ~0.36 s timed: several clock readings
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-path", default="clustered", choices=["clustered", "per-stage"],
                    help="the decode step's path: the clustered step (default; falls back to per-stage launches "
                         "where it does not plan) or the per-stage GEMV launches")
    ap.add_argument("--section", default="all",
                    choices=["all", "decode", "moe", "lm_head", "prefill", "attention", "streams", "gemv",
                             "clustered"],
                    help="moe / lm_head: only the MoE prefill timings / the lm_head GEMV timing "
                         "(for profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    import torch
    import q4synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    shape = q4synth.QWEN3_0P6B
    M = 1
    algo_bytes = shape.weight_bytes_per_step() + 0  # vectors added below
    # activation bytes per step: each GEMV reads its x once and writes y once
    vec = 0
    for nm, N, K in shape.layer_linears():
        vec += M * (K + N) * 2
    vec = shape.n_layers * vec + M * (shape.hidden * 2 + shape.vocab * 4)
    algo_bytes += vec
    config = {"workload": f"{shape.name} decode weight stream, M={M}", "layers": shape.n_layers,
              "hidden": shape.hidden, "q": shape.q, "kv": shape.kv, "ffn": shape.ffn, "vocab": shape.vocab,
              "format": "Q4 group-64, fp16 scale+bias, 8 codes per uint32",
              "bytes_per_step": algo_bytes,
              "l2": "no flush: per-step weight footprint 336.8 MB exceeds the 129 MB L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        host_model = q4synth.decode_weights(shape)
        for _ in range(args.warmup):
            cpu_oracle_rate(shape, host_model, 0, one_sample=True)
        t0 = time.perf_counter()
        total_rate_w = 0.0
        times = []
        for _ in range(args.steps):
            r, _, t = cpu_oracle_rate(shape, host_model, 0, one_sample=True)
            times.append(t)
        wall = time.perf_counter() - t0
        # each step is 1/L of a token's weights
        tok = args.steps / shape.n_layers
        value = tok / sum(times)
        out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sum(times) / args.steps,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic", "config": config,
               "cpu_baseline": {"value": value, "unit": "tok/s", "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": f"per step: one layer's 7 matrices + 1/{shape.n_layers} of lm_head "
                                          f"rows (1/{shape.n_layers} of a token's weights)"},
               "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
               "wall_s": wall}
        print(json.dumps(out))
        return

    import bit_quantized_gemv_q4_gb300 as q4
    from bit_quantized_gemv_q4_gb300 import build as qbuild
    qbuild.build()

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.section == "moe":
        print(json.dumps({"moe_prefill": moe_prefill(device)}))
        return
    if args.section == "streams":
        print(json.dumps({"decode_streams": decode_streams(device)}))
        return
    if args.section == "gemv":
        print(json.dumps({"single_gemv": single_gemv(q4, device)}))
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    if args.section == "lm_head":
        _, dlm, _ = make_model(shape, device, layers=False)
        xl = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4242, M, shape.hidden)).to(device)
        ms_l = lm_head_ms(q4, dlm, xl, M, torch.cuda.current_stream(device), device)
        nb = shape.vocab * shape.hidden * 0.5625 + shape.hidden * 2 + shape.vocab * 4
        peak, peak_kind = peaks()
        print(json.dumps({"lm_head_gemv": {"ms": ms_l, "gbs": nb / (ms_l / 1000.0) / 1e9,
                                           "frac": nb / (ms_l / 1000.0) / 1e9 / peak, "peak_kind": peak_kind,
                                           "shape": f"M={M} N={shape.vocab} K={shape.hidden}, 4 rotating copies"},
                          "lm_head_gemv8": q8_lm_head(q4, device),
                          "lm_head_gemv_bits": bits_lm_head(q4, device)}))
        return
    dl, dlm, host_model = make_model(shape, device)
    if args.section == "prefill":
        print(json.dumps({"dense_prefill": dense_prefill(device, dl, dlm, shape)}))
        return
    if args.section == "attention":
        print(json.dumps({"decode_attention": decode_attention(device, dl, dlm, shape)}))
        return
    if args.section == "clustered":
        xc = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4242, M, shape.hidden)).to(device)
        print(json.dumps({"decode_clustered": decode_clustered(q4, device, dl, dlm, shape, xc, steps=args.steps,
                                                               warmup=args.warmup)}))
        return
    table = q4.LayerTable(dl, dlm, hidden=shape.hidden, M=M,
                          flags=q4.Q4_DECODE_CLUSTERED if args.decode_path == "clustered" else 0)
    nws = q4.q4_decode_workspace_bytes(table)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    table.set_workspace(ws, nws)
    x_host = torch.from_numpy(q4synth.activations(q4synth.BASE_SEED + 4242, M, shape.hidden))
    x = x_host.to(device)
    logits = torch.empty(M, shape.vocab, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        q4.q4_decode_step(table, x, logits, stream)
    st = q4.q4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    path_id = q4.q4_decode_path(table)
    path = "clustered" if path_id == 3 else "per-stage"
    launches_per_step = 3 if path == "clustered" else 4 * shape.n_layers + 1
    config["path"] = ("clustered step: layer stack as one launch of 16-CTA clusters + k/v launch + lm_head "
                      "GEMV (3 launches per step)" if path == "clustered" else
                      f"per-stage GEMV launches ({launches_per_step} per step), graph + PDL")

    # ---- device-resident timed regions: each exactly K steps between a
    # barrier and a synchronisation on both sides, repeated until the regions
    # together last at least 100 ms so the clock samples fall inside them;
    # value = the median region
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    region_ms = []
    with ClockSampler(local) as clk:
        clk.start()
        while True:
            barrier()
            e0.record(stream)
            for _ in range(args.steps):
                q4.q4_decode_step(table, x, logits, stream)
            e1.record(stream)
            barrier()
            region_ms.append(max_over_ranks(e0.elapsed_time(e1), world, device))
            done = sum(region_ms) >= 100.0 or len(region_ms) >= 1000
            if world > 1:  # every rank takes the same number of regions
                flag = torch.tensor([1.0 if done else 0.0], device=device)
                torch.distributed.all_reduce(flag, op=torch.distributed.ReduceOp.MIN)
                done = flag.item() > 0.5
            if done:
                break
        clk.stop()
    ms = statistics.median(region_ms)
    ms_per_step = ms / args.steps
    value = job_rate(world, M, args.steps, ms)

    # ---- end to end through the C ABI with host buffers
    x_pin = x_host.pin_memory()
    out_pin = torch.empty(M, shape.vocab, dtype=torch.float32).pin_memory()
    for _ in range(3):
        x.copy_(x_pin, non_blocking=True)
        q4.q4_decode_step(table, x, logits, stream)
        out_pin.copy_(logits, non_blocking=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        x.copy_(x_pin, non_blocking=True)
        q4.q4_decode_step(table, x, logits, stream)
        out_pin.copy_(logits, non_blocking=True)
    e1.record(stream)
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, device)
    e2e_value = job_rate(world, M, args.steps, ms_e2e)

    lm_ms = lm_head_ms(q4, dlm, x, M, stream, device) if rank == 0 else None
    st = q4.q4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after timing")

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # repetitions of the device-resident step (context beside the headline's
    # single timed region): 5 runs of 200 steps, best and median
    reps = []
    for _ in range(5):
        e0.record(stream)
        for _ in range(200):
            q4.q4_decode_step(table, x, logits, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        reps.append(e0.elapsed_time(e1) / 200)
    reps_status = q4.q4_device_status(stream)

    peak, peak_kind = peaks()
    achieved = algo_bytes / (ms_per_step / 1000.0) / 1e9
    tr = recorded_traffic(path)
    lm_bytes = shape.vocab * shape.hidden * 0.5625 + shape.hidden * 2 + shape.vocab * 4
    out = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "hbm_gbs": achieved, "hbm_frac_of_measured": achieved / peak,
        "hbm_frac_of_nominal": achieved / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind,
                     "kernel": ("q4_step_kernel + q4_step_kv_kernel + q4_gemv_kernel<1> (lm_head): the "
                                "step's 3 launches; achieved = algorithmic bytes per step / step time"
                                if path == "clustered" else
                                "q4_gemv_kernel<1> (all 113 launches of a step; achieved = algorithmic bytes "
                                "per step / step time)"),
                     "traffic": tr[0] if tr else None, "traffic_unit": "DRAM bytes per step (ncu)",
                     "algorithmic_bytes_per_step": algo_bytes},
        "lm_head_gemv": {"ms": lm_ms, "gbs": lm_bytes / (lm_ms / 1000.0) / 1e9 if lm_ms else None,
                         "frac": (lm_bytes / (lm_ms / 1000.0) / 1e9) / peak if lm_ms else None,
                         "shape": f"M={M} N={shape.vocab} K={shape.hidden}, 4 rotating copies"},
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": M * shape.hidden * 2,
                "d2h_bytes_per_step": M * shape.vocab * 4},
        "decode_step_reps": {"runs": 5, "steps_per_run": 200, "ms_best": min(reps),
                             "ms_median": statistics.median(reps), "tok_per_s_best": M * 1000.0 / min(reps),
                             "device_status": reps_status},
        "gpu_launches": launches_per_step * args.steps,
        "timed_regions": {"count": len(region_ms), "steps_each": args.steps, "ms_median": ms,
                          "ms_min": min(region_ms), "ms_max": max(region_ms), "ms_total": sum(region_ms)},
        "clocks": clk.summary(),
    }
    if args.section == "all":
        out["lm_head_gemv8"] = q8_lm_head(q4, device)
        out["lm_head_gemv_bits"] = bits_lm_head(q4, device)
        out["moe_prefill"] = moe_prefill(device)
        out["dense_prefill"] = dense_prefill(device, dl, dlm, shape)
        out["decode_attention"] = decode_attention(device, dl, dlm, shape)
        out["decode_clustered"] = decode_clustered(q4, device, dl, dlm, shape, x)
        out["decode_per_stage"] = decode_per_stage(q4, device, dl, dlm, shape, x)
        out["decode_streams"] = decode_streams(device)
        try:  # context only, measured last; the lines above stand if it fails
            out["single_gemv"] = single_gemv(q4, device)
        except Exception as e:  # noqa: BLE001
            out["single_gemv"] = {"error": f"{type(e).__name__}: {e}"}
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rate, n, t = cpu_oracle_rate(shape, host_model, args.cpu_seconds)
        rate1, n1, t1 = cpu_oracle_rate(shape, host_model, args.cpu_seconds / 4, nthreads=1)
        out["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": oracle.max_threads(), "kind": "oracle",
                               "sample": f"{n} samples of 1/{shape.n_layers} of a token's weights "
                                         f"(one layer + a lm_head row slice), {t:.1f} s",
                               "one_thread": {"value": rate1, "unit": "tok/s", "samples": n1, "seconds": t1}}
    print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
