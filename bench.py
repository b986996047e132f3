#!/usr/bin/env python
"""Benchmark of the block-quantized decode path on GB300.

One step = one decode token through a 60-layer weight sweep shaped like the
gem 31B profile (gem docs/research/architecture.md, "Fixed model profiles"):
per layer the Q4_0 matrices q [5376->8192], k [5376->4096], v [5376->4096]
(stored back to back and read by one launch of 16384 rows, since they share
their input), o [8192->5376], gate/up [5376->21504] (one fused gate+up+GELU
launch) and down [21504->5376], M = 1, with bf16 activations chained from one
matrix to the next (o consumes q's output, standing in for attention).  The 420 weight
matrices (16,164,126,720 bytes, far larger than L2) stay resident in HBM; the
whole step is replayed as one CUDA graph.

Printed (rank 0, one JSON line): effective HBM GB/s of the sweep (algorithmic
bytes / time), tokens/s, the end-to-end rate with the token's activation
copied in from pinned host memory and the result copied back every step, the
roofline of the dominant kernel, SM clocks sampled during the timed region,
the CPU oracle as a baseline, and supplementary per-kernel numbers for the
single-matrix workloads (2048x2048 Q8_0, 21504x5376 Q4_0 and Q4_K, gate+up,
small-M, batched decode, the Q8_0 token table).

``--impl reference`` times the CPU oracle instead (on a bounded sample of the
same workload per step) and prints the same line with ``"impl": "reference"``.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "achieved HBM GB/s (% of GB300 peak) for M=1 Q4_0/Q8_0 matvec; layer-sweep tok/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
LAYERS = 60
SEED = 4
HIDDEN, QDIM, KVDIM, FFN = 5376, 8192, 4096, 21504
# (name, N out, K in, input buffer, output buffer); gate and up share one launch
MATRICES = [("q", QDIM, HIDDEN), ("k", KVDIM, HIDDEN), ("v", KVDIM, HIDDEN), ("o", HIDDEN, QDIM),
            ("gate", FFN, HIDDEN), ("up", FFN, HIDDEN), ("down", HIDDEN, FFN)]
WORKLOAD = "decode weight sweep: 60 layers x Q4_0 {q 5376->8192, k 5376->4096, v 5376->4096 (one launch), " \
           "o 8192->5376, gate/up 5376->21504 fused, down 21504->5376}, M=1, chained bf16 activations"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def weight_bytes(N, K):
    return synth.matrix_bytes("q4_0", N, K)


def sweep_bytes_per_layer():
    """Algorithmic bytes of one layer: every weight byte once, plus activation
    reads and output writes (bf16) of each launch."""
    wb = sum(weight_bytes(N, K) for _, N, K in MATRICES)
    act = 0
    act += 2 * HIDDEN + 2 * QDIM + 2 * 2 * KVDIM                # q, k, v (one launch) read h, write outputs
    act += 2 * QDIM + 2 * HIDDEN                                 # o
    act += 2 * HIDDEN + 2 * FFN                                  # gate+up
    act += 2 * FFN + 2 * HIDDEN                                  # down
    return wb, act


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(torch, ms: float, ws: int, device) -> float:
    """The slowest replica's time: with N > 1 ranks the whole job is done only
    when every rank is (all-reduce MAX over the process group)."""
    if ws == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rates(step_bytes: int, steps: int, ws: int, ms: float):
    """Whole-job GB/s and tokens/s: every rank streams `steps` full steps
    (weak scaling), all within the slowest rank's `ms`."""
    sec = ms * 1e-3
    return step_bytes * steps * ws / sec / 1e9, steps * ws / sec


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured", d
    return 6800.0, "fallback", {}


# Sources whose change voids a kernel's profiled DRAM traffic (device code and
# the host-side launch plan).
KERNEL_SOURCES = {
    "qmv_q4_0": ("qbw_device.cuh", "qbw_internal.h", "tc_common.cuh", "qmv_tc_common.cuh", "qmv_tc.cu", "api.cu"),
    "qmv_gateup_q4_0": ("qbw_device.cuh", "qbw_internal.h", "tc_common.cuh", "qmv_tc_common.cuh", "qmv_tc.cu",
                        "api.cu"),
}
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "qmv_sweep_layer_traffic.txt")


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed: a change of
    comments or layout leaves the compiled kernel, and so its profiled
    traffic, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_weight_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch of ``kernel`` in the sweep, from the committed ncu
    summary (lines ``traffic <kernel> <bytes per launch> <source hash>``), or
    None when the kernel's sources changed since the capture."""
    if kernel not in KERNEL_SOURCES or not os.path.exists(TRAFFIC_SUMMARY):
        return None
    for line in open(TRAFFIC_SUMMARY):
        f = line.split()
        if len(f) == 4 and f[0] == "traffic" and f[1] == kernel:
            return int(f[2]) if f[3] == kernel_source_hash(kernel) else None
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        window = [p for t, p in self.samples if t0 <= t <= t1]
        used = "timed"
        if len(window) < 3:
            window = [p for _, p in self.samples]
            used = "bench"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        sm = [num(p[1]) for p in window if num(p[1]) is not None]
        smax = [num(p[2]) for p in window if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in window:
            for name, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(window), "window": used,
                "power_w_max": max((num(p[3]) or 0.0) for p in window)}


# ------------------------------------------------------------------ GPU arm
class Sweep:
    """The 420 resident weight matrices and the chained activation buffers."""

    def __init__(self, torch, qbw, device, layers=LAYERS):
        self.torch, self.qbw, self.dev = torch, qbw, device
        self.layers = layers
        self.offsets = {}
        total = 0
        for layer in range(layers):
            for mi, (name, N, K) in enumerate(MATRICES):
                self.offsets[(layer, name)] = total
                total += weight_bytes(N, K)
        self.total_weight_bytes = total
        self.w = torch.empty(total, dtype=torch.uint8, device=device)
        bf = torch.bfloat16
        self.h = torch.empty(HIDDEN, dtype=bf, device=device)
        self.qkv = torch.empty(QDIM + 2 * KVDIM, dtype=bf, device=device)
        self.q, self.k, self.v = self.qkv[:QDIM], self.qkv[QDIM:QDIM + KVDIM], self.qkv[QDIM + KVDIM:]
        self.o = torch.empty(HIDDEN, dtype=bf, device=device)
        self.a = torch.empty(FFN, dtype=bf, device=device)
        self.layer0_host = {}
        self._specs = self.specs()

    def fill(self, threads=None):
        import concurrent.futures as cf
        torch = self.torch
        threads = threads or min(16, os.cpu_count() or 1)

        def gen(layer):
            return layer, [synth.q4_0_weights(N, K, seed=SEED, stream=mi, layer=layer)
                           for mi, (_, N, K) in enumerate(MATRICES)]

        t0 = time.time()
        with cf.ThreadPoolExecutor(threads) as ex:
            for layer, mats in ex.map(gen, range(self.layers)):
                for (name, N, K), arr in zip(MATRICES, mats):
                    off = self.offsets[(layer, name)]
                    self.w[off:off + arr.size].copy_(torch.from_numpy(arr))
                    if layer == 0:
                        self.layer0_host[name] = arr
        torch.cuda.synchronize()
        log(f"weights: {self.total_weight_bytes / 1e9:.2f} GB generated and resident in {time.time() - t0:.1f} s")

    def view(self, layer, name):
        N, K = {n: (N, K) for n, N, K in MATRICES}[name]
        off = self.offsets[(layer, name)]
        return self.w[off:off + weight_bytes(N, K)]

    def qkv_view(self, layer):
        """q, k and v of a layer, stored back to back: one [16384, 5376] matrix."""
        off = self.offsets[(layer, "q")]
        return self.w[off:off + weight_bytes(QDIM + 2 * KVDIM, HIDDEN)]

    def specs(self):
        """The step's launches in order, 4 per layer: (kernel, call(stream),
        algorithmic bytes = weights + bf16 activation reads + bf16 writes)."""
        qbw = self.qbw

        def mv(w, x, y, N, K):
            return ("qmv_q4_0", lambda s: qbw.qmv_q4_0(w, x, y, 1, N, K, s), weight_bytes(N, K) + 2 * K + 2 * N)

        out = []
        for layer in range(self.layers):
            out += [mv(self.qkv_view(layer), self.h, self.qkv, QDIM + 2 * KVDIM, HIDDEN),
                    mv(self.view(layer, "o"), self.q, self.o, HIDDEN, QDIM),
                    ("qmv_gateup_q4_0",
                     lambda s, L=layer: qbw.qmv_gateup_q4_0(self.view(L, "gate"), self.view(L, "up"), self.o, self.a,
                                                            1, FFN, HIDDEN, s),
                     2 * weight_bytes(FFN, HIDDEN) + 2 * HIDDEN + 2 * FFN),
                    mv(self.view(layer, "down"), self.a, self.h, HIDDEN, FFN)]
        return out

    def launches(self, stream=None, kernel=None):
        """Enqueue one token (or only the launches of one kernel)."""
        for k, call, _ in self._specs:
            if kernel is None or k == kernel:
                call(stream)

    LAUNCHES_PER_STEP = LAYERS * 4

    def kernel_timing(self, stream, replays):
        """Average launch duration of each kernel as it runs in the sweep: its
        own launches of one step, in step order on the same buffers, captured
        as one graph and replayed on ``stream`` between CUDA events."""
        torch = self.torch
        out = {}
        for kernel in sorted({k for k, _, _ in self._specs}):
            sel = [(c, b) for k, c, b in self._specs if k == kernel]
            g = capture(torch, lambda: self.launches(None, kernel), stream)
            time_graph(torch, g, 2, stream)
            ms = time_graph(torch, g, replays, stream) / replays
            out[kernel] = {"launches": len(sel), "bytes": sum(b for _, b in sel), "ms": ms}
            del g
        return out


def time_graph(torch, graph, steps, stream):
    """Replay ``graph`` ``steps`` times on ``stream``; events on the same stream."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()                      # warm every kernel outside capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def supplementary_kernels(torch, qbw, hbm_peak):
    """Single-matrix workloads, each cycled over rotating weight copies whose
    total exceeds twice the L2 size, replayed from a CUDA graph."""
    dev = torch.device("cuda")
    res = {}
    l2 = torch.cuda.get_device_properties(0).L2_cache_size

    def bf16(a):
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    def run(name, nbytes_call, copies, make_call, flops=None):
        calls = [make_call(i) for i in range(copies)]
        s = torch.cuda.Stream()
        g = capture(torch, lambda: [c() for c in calls], s)
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
        reps = max(3, int(2e9 / (nbytes_call * copies)))
        ms = time_graph(torch, g, reps, s)
        us = ms * 1e3 / (reps * copies)
        gbs = nbytes_call / (us * 1e3)
        entry = {"us_per_call": round(us, 3), "GB_per_s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
                 "frac_of_8TBps": round(gbs / NOMINAL_HBM_GBS, 4), "bytes_per_call": nbytes_call,
                 "weight_copies": copies, "rotating_bytes": nbytes_call * copies, "l2_bytes": l2}
        if flops:
            entry["TFLOP_per_s"] = round(flops / (us * 1e-6) / 1e12, 2)
        res[name] = entry
        log(f"{name}: {us:.2f} us/call  {gbs:.0f} GB/s")

    # 2048 x 2048 Q8_0, fp32 in/out
    N = K = 2048
    w = torch.from_numpy(synth.q8_0_weights(N, K, seed=0)).to(dev)
    copies = max(2, int(np.ceil(2.2 * l2 / w.numel())))
    ws = [w.clone() for _ in range(copies)]
    x = torch.from_numpy(synth.activations(K, seed=0)).to(dev)
    y = torch.empty(N, device=dev)
    run("qmv_q8_0 2048x2048 f32", w.numel() + 4 * K + 4 * N, copies,
        lambda i: (lambda: qbw.qmv_q8_0(ws[i], x, y, 1, N, K)))
    del ws, w
    # 21504 x 5376 Q4_0, fp32 in/out
    N, K = 21504, 5376
    w = torch.from_numpy(synth.q4_0_weights(N, K, seed=1)).to(dev)
    copies = max(2, int(np.ceil(2.2 * l2 / w.numel())))
    ws = [w.clone() for _ in range(copies)]
    x = torch.from_numpy(synth.activations(K, seed=1)).to(dev)
    y = torch.empty(N, device=dev)
    run("qmv_q4_0 21504x5376 f32", w.numel() + 4 * K + 4 * N, copies,
        lambda i: (lambda: qbw.qmv_q4_0(ws[i], x, y, 1, N, K)))
    # the same matrix with bf16 activations (the sweep's case), fp32 out
    xb1 = bf16(synth.activations(K, seed=1, dtype="bf16"))
    run("qmv_q4_0 21504x5376 bf16->f32", w.numel() + 2 * K + 4 * N, copies,
        lambda i: (lambda: qbw.qmv_q4_0(ws[i], xb1, y, 1, N, K)))
    # gate+up on two such matrices, bf16 in, fp32 out
    wu = torch.from_numpy(synth.q4_0_weights(N, K, seed=2, stream=1)).to(dev)
    wus = [wu.clone() for _ in range(copies)]
    xb = bf16(synth.activations(K, seed=2, dtype="bf16"))
    run("qmv_gateup_q4_0 2x21504x5376 bf16->f32", 2 * w.numel() + 2 * K + 4 * N, copies,
        lambda i: (lambda: qbw.qmv_gateup_q4_0(ws[i], wus[i], xb, y, 1, N, K)))
    del ws, wus, w, wu
    # the same shape in Q4_K (256-weight super-blocks, 144 bytes each), fp32 in/out
    N, K = 21504, 5376
    w = torch.from_numpy(synth.q4_k_weights(N, K, seed=1)).to(dev)
    copies = max(2, int(np.ceil(2.2 * l2 / w.numel())))
    ws = [w.clone() for _ in range(copies)]
    x = torch.from_numpy(synth.activations(K, seed=1)).to(dev)
    y = torch.empty(N, device=dev)
    run("qmv_q4_k 21504x5376 f32", w.numel() + 4 * K + 4 * N, copies,
        lambda i: (lambda: qbw.qmv_q4_k(ws[i], x, y, 1, N, K)))
    xk = bf16(synth.activations(K, seed=1, dtype="bf16"))
    run("qmv_q4_k 21504x5376 bf16->f32", w.numel() + 2 * K + 4 * N, copies,
        lambda i: (lambda: qbw.qmv_q4_k(ws[i], xk, y, 1, N, K)))
    del ws, w
    # the down projection 5376 x 21504 (Q4_0, bf16 -> bf16) on a GELU(g) * u
    # activation with g, u ~ N(0, 6.6^2), the spread the sweep's first layer
    # produces: most of its elements sit far below their block's largest, so
    # the 8-bit form's error check runs on every unit
    N, K = 5376, 21504
    w = torch.from_numpy(synth.q4_0_weights(N, K, seed=20)).to(dev)
    copies = max(2, int(np.ceil(2.2 * l2 / w.numel())))
    ws = [w.clone() for _ in range(copies)]
    grng = np.random.default_rng(5)
    gg, uu = grng.standard_normal(K) * 6.6, grng.standard_normal(K) * 6.6
    act = 0.5 * gg * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (gg + 0.044715 * gg ** 3))) * uu
    xg = bf16(synth.f32_to_bf16_bits(act.astype(np.float32)))
    xn = bf16(synth.activations(K, seed=20, dtype="bf16"))
    yb = torch.empty(N, dtype=torch.bfloat16, device=dev)
    run("qmv_q4_0 5376x21504 bf16->bf16 N(0,1) x", w.numel() + 2 * K + 2 * N, copies,
        lambda i: (lambda: qbw.qmv_q4_0(ws[i], xn, yb, 1, N, K)))
    run("qmv_q4_0 5376x21504 bf16->bf16 GELU(g)*u x", w.numel() + 2 * K + 2 * N, copies,
        lambda i: (lambda: qbw.qmv_q4_0(ws[i], xg, yb, 1, N, K)))
    del ws, w
    # the mixed-bit formats (int2-symmetric, int4-affine, int8), 21504 x 5376:
    # groups of 32, bf16 -> fp32 and fp32 -> fp32 (the tensor-core forms), and
    # groups of 16, bf16 -> fp32 (the CUDA-core kernel)
    N, K = 21504, 5376
    xm = bf16(synth.activations(K, seed=9, dtype="bf16"))
    xm32 = torch.from_numpy(synth.activations(K, seed=9)).to(dev)
    y = torch.empty(N, device=dev)
    for bits in (2, 4, 8):
        name = {2: "int2-symmetric", 4: "int4-affine", 8: "int8"}[bits]
        for G in (32, 16):
            qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=9)
            nbytes = synth.mixbit_bytes(bits, N, K, G)
            copies = max(2, int(np.ceil(2.2 * l2 / nbytes)))
            mats = [(torch.from_numpy(qp.view(np.uint8).copy()).to(dev),
                     torch.from_numpy(sc.view(np.uint8).copy()).to(dev),
                     torch.from_numpy(bi.view(np.uint8).copy()).to(dev) if bi is not None else None)
                    for _ in range(copies)]
            if G == 32:
                run(f"qmv_mixbit {name} {N}x{K} G={G} bf16->f32", nbytes + 2 * K + 4 * N, copies,
                    lambda i, mats=mats, bits=bits, G=G: (lambda: qbw.qmv_mixbit(bits, *mats[i], G, xm, y, 1, N, K)))
                run(f"qmv_mixbit {name} {N}x{K} G={G} f32->f32", nbytes + 4 * K + 4 * N, copies,
                    lambda i, mats=mats, bits=bits, G=G: (lambda: qbw.qmv_mixbit(bits, *mats[i], G, xm32, y, 1, N, K)))
            else:
                run(f"qmv_mixbit {name} {N}x{K} G={G} bf16->f32 (CUDA cores)", nbytes + 2 * K + 4 * N, copies,
                    lambda i, mats=mats, bits=bits, G=G: (lambda: qbw.qmv_mixbit(bits, *mats[i], G, xm, y, 1, N, K)))
            del mats
    # small-M tiles
    for (N, K) in ((5376, 5376), (5376, 21504)):
        w = torch.from_numpy(synth.q4_0_weights(N, K, seed=3)).to(dev)
        copies = max(2, int(np.ceil(2.2 * l2 / w.numel())))
        ws = [w.clone() for _ in range(copies)]
        for M in (8, 16, 32):
            X = bf16(synth.activations((M, K), seed=3, dtype="bf16"))
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsb = qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K)
            work = torch.zeros(max(wsb, 1), dtype=torch.uint8, device=dev)
            run(f"qmm_q4_0_smallM M={M} {N}x{K} bf16", w.numel() + 2 * M * K + 2 * M * N, copies,
                lambda i, X=X, Y=Y, M=M, N=N, K=K, work=work: (lambda: qbw.qmm_q4_0_smallM(ws[i], X, Y, M, N, K, work)),
                flops=2.0 * M * N * K)
        del ws, w
    # batched decode: M = 2 and 4 sequences sharing one read of the q|k|v and
    # down weights (the tensor-core small-M path)
    for (N, K) in ((16384, 5376), (5376, 21504)):
        w = torch.from_numpy(synth.q4_0_weights(N, K, seed=5)).to(dev)
        copies = max(2, int(np.ceil(2.2 * l2 / w.numel())))
        ws = [w.clone() for _ in range(copies)]
        for M in (2, 4):
            X = bf16(synth.activations((M, K), seed=5, dtype="bf16"))
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsb = qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K)
            work = torch.zeros(max(wsb, 1), dtype=torch.uint8, device=dev)
            run(f"batched decode qmm_q4_0_smallM M={M} {N}x{K} bf16", w.numel() + 2 * M * K + 2 * M * N, copies,
                lambda i, X=X, Y=Y, M=M, N=N, K=K, work=work: (lambda: qbw.qmm_q4_0_smallM(ws[i], X, Y, M, N, K, work)))
        del ws, w
    # the Q8_0 token table of the 31B profile (262144 x 5376, 1.5 GB, larger
    # than L2): tied LM head matvec, and the embedding-row gather of a token
    N, K = 262144, 5376
    w = torch.from_numpy(synth.q8_0_weights(N, K, seed=12)).to(dev)
    xb = bf16(synth.activations(K, seed=12, dtype="bf16"))
    y = torch.empty(N, device=dev)
    run("qmv_q8_0 262144x5376 bf16->f32 (token table as LM head)", w.numel() + 2 * K + 4 * N, 1,
        lambda i: (lambda: qbw.qmv_q8_0(w, xb, y, 1, N, K)))
    for n_ids in (1, 32):
        ids = torch.from_numpy(np.arange(0, N, N // n_ids, dtype=np.int32)[:n_ids]).to(dev)
        out = torch.empty(n_ids, K, dtype=torch.bfloat16, device=dev)
        run(f"qembed_q8_0 {n_ids} rows of 262144x5376 -> bf16", n_ids * (K // 32 * 34 + 2 * K) + 4 * n_ids, 1,
            lambda i, ids=ids, out=out: (lambda: qbw.qembed_q8_0(w, ids, out, N, K)))
    del w
    torch.cuda.empty_cache()
    return res


def host_cpu():
    """The host's CPU model (lscpu, else /proc/cpuinfo) and the size of this
    process's CPU affinity set."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return model or "unknown", len(os.sched_getaffinity(0))


def cpu_sweep_sample(layer0_host, x_bits, budget_s, threads):
    """The oracle, as it stands, on a bounded sample of the sweep: layer 0's
    seven matrices in order, in chunks of rows, repeated until ``budget_s``
    elapse; ``threads``: its OpenMP build over all cores."""
    import oracle
    rng = np.random.default_rng(0)
    xs = {name: (x_bits if name in ("q", "k", "v") else
                 synth.f32_to_bf16_bits(rng.standard_normal(K).astype(np.float32)))
          for name, N, K in MATRICES}
    chunk = 4096 if threads else 256
    done_bytes = 0
    t0 = time.time()
    while time.time() - t0 < budget_s:
        for name, N, K in MATRICES:
            rb = synth.row_bytes("q4_0", K)
            for n in range(0, N, chunk):
                n1 = min(N, n + chunk)
                oracle.qmv_rows("q4_0", layer0_host[name], xs[name], n, n1, K, threads=threads)
                done_bytes += (n1 - n) * rb
                if time.time() - t0 >= budget_s:
                    break
            if time.time() - t0 >= budget_s:
                break
    dt = time.time() - t0
    return done_bytes / dt / 1e9, dt, done_bytes, done_bytes / sum(weight_bytes(N, K) for _, N, K in MATRICES)


def cpu_configs():
    """The oracle's time per call on configs 1 to 4 (one thread and all
    cores), best of two calls; the small-M tile at M = 8 (the oracle's cost
    grows linearly in M)."""
    import oracle
    res = {}

    def timed(name, nbytes, fn):
        for threads in (False, True):
            dt = 1e30
            for _ in range(2):              # best of two (the first all-core call starts the thread pool)
                t0 = time.perf_counter()
                fn(threads)
                dt = min(dt, time.perf_counter() - t0)
            res.setdefault(name, {})["all_cores" if threads else "one_thread"] = {
                "us_per_call": round(dt * 1e6, 1), "GB_per_s": round(nbytes / dt / 1e9, 4)}

    N = K = 2048
    w, x = synth.q8_0_weights(N, K, seed=0), synth.activations(K, seed=0)
    timed("config 1: qmv_q8_0 2048x2048 f32", w.size + 8 * K,
          lambda t: oracle.qmv_rows("q8_0", w, x, 0, N, K, threads=t))
    N, K = 21504, 5376
    w, x = synth.q4_0_weights(N, K, seed=1), synth.activations(K, seed=1)
    timed("config 2: qmv_q4_0 21504x5376 f32", w.size + 4 * K + 4 * N,
          lambda t: oracle.qmv_rows("q4_0", w, x, 0, N, K, threads=t))
    wu, xb = synth.q4_0_weights(N, K, seed=2, stream=1), synth.activations(K, seed=2, dtype="bf16")
    timed("config 3: gateup_q4_0 2x21504x5376 bf16", 2 * w.size + 2 * K + 4 * N,
          lambda t: oracle.gateup_q4_0(w, wu, xb, N, K, threads=t))
    for (N, K) in ((5376, 5376), (5376, 21504)):
        w, X = synth.q4_0_weights(N, K, seed=3), synth.activations((8, K), seed=3, dtype="bf16")
        timed(f"config 4: qmm_q4_0 M=8 {N}x{K} bf16", w.size + 2 * 8 * (K + N),
              lambda t: oracle.qmm_q4_0(w, X, 8, N, K, threads=t))
    return res


def cpu_baseline(layer0_host, x_bits, budget_s):
    """The CPU oracle as the reported baseline: the sweep sample on all cores
    (the OpenMP build) and on one thread, the host's CPU, and per-config
    times."""
    import oracle
    oracle.lib()
    model, cores = host_cpu()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    one = cpu_sweep_sample(layer0_host, x_bits, budget_s / 2, threads=False)
    try:
        oracle.lib_mt()
        allc = cpu_sweep_sample(layer0_host, x_bits, budget_s / 2, threads=True)
    except (OSError, subprocess.CalledProcessError) as e:
        log(f"OpenMP oracle unavailable: {e}")
        allc = None
    base = allc or one
    out = {"value": round(base[0], 4), "unit": UNIT, "cores": cores if allc else 1, "kind": "oracle",
           "sample": f"oracle qmv_q4_0 over layer 0's seven matrices, {base[3]:.2f} passes ({base[2]} weight "
                     f"bytes) in {base[1]:.1f} s, {'all ' + str(cores) + ' cores (OpenMP over rows)' if allc else 'one thread'}",
           "cpu_model": model, "affinity_cpus": cores,
           "one_thread": {"value": round(one[0], 4), "unit": UNIT, "cores": 1,
                          "sample": f"{one[3]:.2f} passes in {one[1]:.1f} s"}}
    try:
        out["per_config"] = cpu_configs()
    except Exception as e:     # the baseline is reported, never required
        log(f"per-config oracle timing failed: {e}")
    return out


def gpu_arm(args):
    import torch
    import block_quantized_weight_gb300 as qbw

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    qbw.load()
    hbm_peak, peak_kind, peaks = load_peaks()

    sweep = Sweep(torch, qbw, dev)
    sweep.fill()
    x0 = synth.activations(HIDDEN, seed=SEED, dtype="bf16")
    x0_dev = torch.from_numpy(x0.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    sweep.h.copy_(x0_dev)

    stream = torch.cuda.Stream()

    def step():
        sweep.launches()

    graph = capture(torch, step, stream)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = str(getattr(props, "uuid", ""))
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else "0"))
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            sweep.h.copy_(x0_dev)
            graph.replay()
        sweep.h.copy_(x0_dev)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    t_start = time.time()
    ms = time_graph(torch, graph, args.steps, stream)
    t_end = time.time()
    ms = max_over_ranks(torch, ms, ws, dev)
    assert qbw.fault_read(clear=True, stream=stream) == 0, "a kernel recorded a fault"

    # end to end: the token's activation in from pinned host memory, the
    # step's result out to pinned host memory, every step
    h_in = torch.from_numpy(x0.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    h_out = torch.empty(HIDDEN, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(50, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):                # untimed: the first host copies of the pinned buffers
            sweep.h.copy_(h_in, non_blocking=True)
            graph.replay()
            h_out.copy_(sweep.h, non_blocking=True)
            stream.synchronize()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            sweep.h.copy_(h_in, non_blocking=True)
            graph.replay()
            h_out.copy_(sweep.h, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0
    per_kernel = sweep.kernel_timing(stream, replays=max(5, min(args.steps, 50)))
    clocks.stop()
    assert qbw.fault_read(clear=True, stream=stream) == 0, "a kernel recorded a fault"

    wb, ab = sweep_bytes_per_layer()
    step_bytes = LAYERS * (wb + ab)
    value, tok_s = job_rates(step_bytes, args.steps, ws, ms)
    e2e_value = step_bytes * e2e_steps * ws / e2e_s / 1e9

    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    pk = per_kernel[dom]
    achieved = pk["bytes"] / (pk["ms"] * 1e-3) / 1e9
    step_ms = ms / args.steps
    traffic = profiled_traffic(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "peak_kind": f"{peak_kind} copy bandwidth (hbm_gbs)",
                "frac_of_8TBps": round(achieved / NOMINAL_HBM_GBS, 4),
                "bytes_per_launch": round(pk["bytes"] / pk["launches"]), "launches": pk["launches"],
                "us_per_launch": round(pk["ms"] / pk["launches"] * 1e3, 3),
                "traffic": traffic,
                "share_of_step": {k: round(v["ms"] / step_ms, 4) for k, v in per_kernel.items()},
                "measured": "the kernel's own launches of one step, in step order on the sweep's buffers, captured "
                            "as one CUDA graph and replayed between CUDA events on the launching stream"}
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    supp = {} if args.no_kernels else supplementary_kernels(torch, qbw, hbm_peak)
    chained = {} if args.no_kernels else sweep_as_chain(torch, qbw, sweep, x0_dev, stream, graph, step_bytes)
    cpu = None
    if not args.no_cpu and ws == 1:
        cpu = cpu_baseline(sweep.layer0_host, x0, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": LAYERS, "bytes_per_step": step_bytes,
                   "weight_bytes_per_step": LAYERS * wb, "tok_per_s": round(tok_s, 2),
                   "frac_of_measured_hbm": round(value / hbm_peak, 4), "frac_of_8TBps": round(value / NOMINAL_HBM_GBS, 4),
                   "l2": "inputs larger than L2: 16.16 GB of weights streamed per step, no flush needed",
                   "parallelism": "replicas" if ws > 1 else "single GPU", "graph": "one CUDA graph per step",
                   "seed": SEED},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "tok_per_s": round(e2e_steps * ws / e2e_s, 2),
                "h2d_bytes_per_step": 2 * HIDDEN, "d2h_bytes_per_step": 2 * HIDDEN, "steps": e2e_steps,
                "path": "pinned host -> device copy, graph replay of the C-ABI launches, device -> pinned host copy, "
                        "stream sync, every step"},
        "gpu_launches": Sweep.LAUNCHES_PER_STEP * args.steps,
        "roofline": roofline,
        "clocks": clocks.summary(t_start - 0.05, t_end + 0.05),
        "cpu_baseline": cpu,
        "kernels": supp,
        "sweep_as_one_launch": chained.get("sweep_as_one_launch"),
        "sweep_as_prefetching_launches": chained.get("sweep_as_prefetching_launches"),
        "per_kernel_in_sweep": {k: {"launches": v["launches"], "ms": round(v["ms"], 4),
                                    "GB_per_s": round(v["bytes"] / (v["ms"] * 1e-3) / 1e9, 1)}
                                for k, v in per_kernel.items()},
        "gpu": torch.cuda.get_device_name(),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def sweep_chain_steps(sweep):
    """The sweep's 240 launches as chain steps, on the sweep's own buffers."""
    steps = []
    for L in range(sweep.layers):
        steps += [(sweep.qkv_view(L), None, sweep.h, sweep.qkv, QDIM + 2 * KVDIM, HIDDEN),
                  (sweep.view(L, "o"), None, sweep.q, sweep.o, HIDDEN, QDIM),
                  (sweep.view(L, "gate"), sweep.view(L, "up"), sweep.o, sweep.a, FFN, HIDDEN),
                  (sweep.view(L, "down"), None, sweep.a, sweep.h, HIDDEN, FFN)]
    return steps


def sweep_as_chain(torch, qbw, sweep, x0_dev, stream, graph, step_bytes, replays=50):
    """The same token through a chain over the sweep's 240 steps and buffers,
    in its two forms: one cooperative launch with a grid barrier between steps
    (qbw_chain_run), and one launch per step in which each launch prefetches
    the next step's first weight tiles into L2 (qbw_chain_run_launches).  For
    each, its time and whether its final activation equals the graph of 240
    separate launches bit for bit."""
    chain = qbw.Chain(sweep_chain_steps(sweep))
    forms = {"sweep_as_one_launch": (chain.run, 1, "qbw_chain_run: the 240 steps as one cooperative launch "
                                                   "with a grid barrier between steps"),
             "sweep_as_prefetching_launches": (chain.run_launches, Sweep.LAUNCHES_PER_STEP,
                                               "qbw_chain_run_launches: one launch per step, each prefetching "
                                               "the next step's first weight tiles into L2")}
    out = {}
    try:
        with torch.cuda.stream(stream):
            sweep.h.copy_(x0_dev)
            graph.replay()
            h_graph = sweep.h.clone()
        for key, (run, launches, what) in forms.items():
            with torch.cuda.stream(stream):
                sweep.h.copy_(x0_dev)
                run(stream)
            torch.cuda.synchronize()
            same = bool(torch.equal(h_graph.view(torch.int16), sweep.h.view(torch.int16)))
            g = capture(torch, lambda: run(torch.cuda.current_stream()), stream)
            time_graph(torch, g, 3, stream)
            ms = time_graph(torch, g, replays, stream) / replays
            assert qbw.fault_read(clear=True, stream=stream) == 0, f"{key} recorded a fault"
            out[key] = {"ms_per_step": round(ms, 4), "GB_per_s": round(step_bytes / (ms * 1e-3) / 1e9, 1),
                        "tok_per_s": round(1e3 / ms, 2), "final_activation_bit_identical_to_graph": same,
                        "launches_per_step": launches, "what": what}
    finally:
        chain.close()
    return out


def profile_case(args):
    """A small, self-contained run for profiler captures: the single-matrix
    workload named by --profile, ``warmup + steps`` calls over a few rotating
    weight copies (well under 1 GB on the device), or ``--profile sweep``: the
    sweep's own launches over 6 layers (1.6 GB), 36 launches per call."""
    import torch
    import block_quantized_weight_gb300 as qbw
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    qbw.load()
    name = args.profile
    copies = 4
    if name == "q8_0":
        # 2048 x 2048 (4.5 MB) over 64 rotating copies (285 MB, larger than L2)
        N = K = 2048
        copies = 64
        w0 = torch.from_numpy(synth.q8_0_weights(N, K, seed=0)).to(dev)
        ws = [w0.clone() for _ in range(copies)]
        x = torch.from_numpy(synth.activations(K, seed=0)).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_q8_0(ws[i % copies], x, y, 1, N, K)
        nbytes = ws[0].numel() + 4 * K + 4 * N
    elif name == "q8_0_lmhead":
        # the 262144 x 5376 Q8_0 token table as LM head (1.5 GB), bf16 x
        N, K = 262144, 5376
        ws = [torch.from_numpy(synth.q8_0_weights(N, K, seed=12)).to(dev)]
        xb = torch.from_numpy(synth.activations(K, seed=12, dtype="bf16").view(np.int16).copy()).view(
            torch.bfloat16).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_q8_0(ws[0], xb, y, 1, N, K)
        nbytes = ws[0].numel() + 2 * K + 4 * N
    elif name == "q4_0":
        N, K = 21504, 5376
        ws = [torch.from_numpy(synth.q4_0_weights(N, K, seed=1)).to(dev) for _ in range(copies)]
        x = torch.from_numpy(synth.activations(K, seed=1)).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_q4_0(ws[i % copies], x, y, 1, N, K)
        nbytes = ws[0].numel() + 4 * K + 4 * N
    elif name == "q4_0_bf16":
        # the same matrix with bf16 activations: the tensor-core kernel's 8-bit operand form
        N, K = 21504, 5376
        ws = [torch.from_numpy(synth.q4_0_weights(N, K, seed=1)).to(dev) for _ in range(copies)]
        xb = torch.from_numpy(synth.activations(K, seed=1, dtype="bf16").view(np.int16).copy()).view(
            torch.bfloat16).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_q4_0(ws[i % copies], xb, y, 1, N, K)
        nbytes = ws[0].numel() + 2 * K + 4 * N
    elif name == "q4_0_stream":
        # 4096 x 5376 Q4_0 (12.4 MB, below the tensor-core threshold): the
        # streaming kernel, over 25 rotating copies (310 MB, larger than L2)
        N, K = 4096, 5376
        copies = 25
        ws = [torch.from_numpy(synth.q4_0_weights(N, K, seed=1)).to(dev) for _ in range(copies)]
        x = torch.from_numpy(synth.activations(K, seed=1)).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_q4_0(ws[i % copies], x, y, 1, N, K)
        nbytes = ws[0].numel() + 4 * K + 4 * N
    elif name == "qmm2_qkv":
        # two tokens over the 16384 x 5376 q|k|v matrix (49.5 MB): the
        # tensor-core M = 1 kernel's bf16-code form, both tokens in one B
        N, K, M = 16384, 5376, 2
        copies = 7
        ws = [torch.from_numpy(synth.q4_0_weights(N, K, seed=3)).to(dev) for _ in range(copies)]
        X = torch.from_numpy(synth.activations((M, K), seed=3, dtype="bf16").view(np.int16).copy()).view(
            torch.bfloat16).to(dev)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        work = torch.zeros(256, dtype=torch.uint8, device=dev)
        call = lambda i: qbw.qmm_q4_0_smallM(ws[i % copies], X, Y, M, N, K, work)
        nbytes = ws[0].numel() + 2 * M * K + 2 * M * N
    elif name == "q4_k":
        N, K = 21504, 5376
        ws = [torch.from_numpy(synth.q4_k_weights(N, K, seed=1)).to(dev) for _ in range(copies)]
        x = torch.from_numpy(synth.activations(K, seed=1)).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_q4_k(ws[i % copies], x, y, 1, N, K)
        nbytes = ws[0].numel() + 4 * K + 4 * N
    elif name == "gateup":
        N, K = 21504, 5376
        wg = [torch.from_numpy(synth.q4_0_weights(N, K, seed=2, stream=0)).to(dev) for _ in range(2)]
        wu = [torch.from_numpy(synth.q4_0_weights(N, K, seed=2, stream=1)).to(dev) for _ in range(2)]
        xb = torch.from_numpy(synth.activations(K, seed=2, dtype="bf16").view(np.int16).copy()).view(
            torch.bfloat16).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_gateup_q4_0(wg[i % 2], wu[i % 2], xb, y, 1, N, K)
        nbytes = 2 * wg[0].numel() + 2 * K + 4 * N
    elif name == "chain":
        # the sweep's steps over 2 layers as one cooperative chain launch
        sweep = Sweep(torch, qbw, dev, layers=2)
        sweep.fill()
        sweep.h.copy_(torch.from_numpy(synth.activations(HIDDEN, seed=SEED, dtype="bf16").view(np.int16).copy())
                      .view(torch.bfloat16).to(dev))
        chain = qbw.Chain(sweep_chain_steps(sweep))
        call = lambda i: chain.run()
        nbytes = sum(b for _, _, b in sweep._specs)
    elif name == "sweep":
        # the sweep's own launches over a few layers (1.6 GB of weights)
        sweep = Sweep(torch, qbw, dev, layers=6)
        sweep.fill()
        sweep.h.copy_(torch.from_numpy(synth.activations(HIDDEN, seed=SEED, dtype="bf16").view(np.int16).copy())
                      .view(torch.bfloat16).to(dev))
        call = lambda i: sweep.launches()
        nbytes = sum(b for _, _, b in sweep._specs)
    elif name.startswith("mixbit"):
        # one mixed-bit matrix, 21504 x 5376, groups of 32, bf16 x (the
        # tensor-core forms), rotating copies larger than L2 together; with the
        # suffix "_f32", fp32 x (the tensor-core forms' three-piece variant);
        # with "_g16", groups of 16 (the CUDA-core kernel)
        f32x = name.endswith("_f32")
        bits = int(name[len("mixbit"):].replace("_f32", "").replace("_g16", ""))
        N, K, G = 21504, 5376, (16 if name.endswith("_g16") else 32)
        qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=9)
        nb = synth.mixbit_bytes(bits, N, K, G)
        copies = max(2, int(np.ceil(300e6 / nb)))
        mats = [(torch.from_numpy(qp.view(np.uint8).copy()).to(dev), torch.from_numpy(sc.view(np.uint8).copy()).to(dev),
                 torch.from_numpy(bi.view(np.uint8).copy()).to(dev) if bi is not None else None) for _ in range(copies)]
        if f32x:
            xb = torch.from_numpy(synth.activations(K, seed=9)).to(dev)
        else:
            xb = torch.from_numpy(synth.activations(K, seed=9, dtype="bf16").view(np.int16).copy()).view(
                torch.bfloat16).to(dev)
        y = torch.empty(N, device=dev)
        call = lambda i: qbw.qmv_mixbit(bits, *mats[i % copies], G, xb, y, 1, N, K)
        nbytes = nb + (4 if f32x else 2) * K + 4 * N
    elif name in ("qmm", "qmm8", "qmm8_5376"):
        # M = 32 (whole-tile splits) or M = 8 (stream-K) over 5376 x 21504, or
        # M = 8 over 5376 x 5376 (cluster splits)
        M, N, K = {"qmm": (32, 5376, 21504), "qmm8": (8, 5376, 21504), "qmm8_5376": (8, 5376, 5376)}[name]
        copies = max(copies, int(np.ceil(300e6 / (N * K // 32 * 18))))
        ws = [torch.from_numpy(synth.q4_0_weights(N, K, seed=3)).to(dev) for _ in range(copies)]
        X = torch.from_numpy(synth.activations((M, K), seed=3, dtype="bf16").view(np.int16).copy()).view(
            torch.bfloat16).to(dev)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        work = torch.zeros(max(1, qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K)), dtype=torch.uint8, device=dev)
        call = lambda i: qbw.qmm_q4_0_smallM(ws[i % copies], X, Y, M, N, K, work)
        nbytes = ws[0].numel() + 2 * M * K + 2 * M * N
    else:
        raise SystemExit(f"unknown --profile case {name}")
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        call(args.warmup + i)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    assert qbw.fault_read(clear=True) == 0, "a kernel recorded a fault"
    print(json.dumps({"profile_case": name, "calls": args.steps, "us_per_call": round(us, 3),
                      "GB_per_s": round(nbytes / (us * 1e3), 1)}), flush=True)


# ------------------------------------------------------------------ reference arm
def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.lib()
    model, cores = host_cpu()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    try:
        oracle.lib_mt()
        threads = True
    except (OSError, subprocess.CalledProcessError):
        threads, cores = False, 1
    # one layer's first matrices, regenerated exactly as the GPU arm does
    mats = {name: synth.q4_0_weights(N, K, seed=SEED, stream=mi, layer=0) for mi, (name, N, K) in enumerate(MATRICES)
            if name in ("q", "k", "v")}
    x = synth.activations(HIDDEN, seed=SEED, dtype="bf16")
    rb = synth.row_bytes("q4_0", HIDDEN)
    # size one step so that warmup + steps stay within about two minutes
    t0 = time.time()
    oracle.qmv_rows("q4_0", mats["q"], x, 0, 1024, HIDDEN, threads=threads)
    per_row = (time.time() - t0) / 1024
    step_s = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    rows = max(8, int(step_s / per_row))
    rows = min(rows, QDIM)

    def one_step():
        oracle.qmv_rows("q4_0", mats["q"], x, 0, rows, HIDDEN, threads=threads)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    nbytes = rows * rb
    value = nbytes * args.steps / dt / 1e9
    sample = (f"oracle qmv_q4_0 on the first {rows} rows of layer 0's q matrix (5376 inputs) per step, "
              + (f"all {cores} cores of the host ({model}; OpenMP over rows)" if threads else "one thread"))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_bytes_per_step": nbytes},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                             "cpu_model": model, "affinity_cpus": len(os.sched_getaffinity(0))},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["qbw", "reference"], default="qbw")
    ap.add_argument("--no-kernels", action="store_true", help="skip the single-matrix supplementary numbers")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile", choices=["q8_0", "q8_0_lmhead", "q4_0", "q4_0_bf16", "q4_k", "gateup", "qmm", "sweep",
                                          "mixbit2", "mixbit4", "mixbit8", "mixbit2_f32", "mixbit4_f32",
                                          "mixbit8_f32", "mixbit2_g16", "mixbit4_g16", "mixbit8_g16", "qmm8", "qmm8_5376", "q4_0_stream",
                                          "qmm2_qkv", "chain"],
                    help="run only one small case (for profiler captures): a single-matrix workload, or the "
                         "sweep's launches over 6 layers")
    args = ap.parse_args()
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != ws and not args.profile:
        ap.error(f"--gpus {args.gpus} needs {args.gpus} processes (launch with torchrun --nproc-per-node "
                 f"{args.gpus}); this run has WORLD_SIZE={ws}")
    if args.profile:
        profile_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
