#!/usr/bin/env python3
"""Benchmark of the attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:

* packed causal GQA prefill of the concurrent Prefill-Only batch (240
  sequences, lengths uniform in [64, 1024], 16 query / 8 KV heads, head_dim
  128) for 28 layers, each layer an independent Q/K/V set (28 x 1.6 GB, so
  every layer's inputs come from HBM, not L2);
* the long-prompt wide beam decode (prompt 1024, W = 400, 5 steps) and the
  short-prompt beam decode (prompt 96, W = 100, 4 steps): per step the
  shared-prefix decode attention with suffix reorder, then the two-stage
  candidate selection over 151,936 bf16 logits.

The headline value is the prefill attention throughput in TFLOP/s (logical
FLOPs of the causal attention, 4 * D * L(L+1)/2 per sequence and query head,
FMA = 2); the decode steps are reported beside it in microseconds and as a
fraction of HBM bandwidth.  Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_packed_varlen_gb300 import workloads as wl  # noqa: E402

METRIC = "packed-prefill attn TFLOPS (% BF16 peak); beam-decode step us (% HBM BW)"
UNIT = "TFLOP/s"
PREFILL_WL = wl.CONCURRENT_PREFILL_BATCH
BEAM_WLS = (wl.LONG_PROMPT_WIDE_BEAM, wl.SHORT_PROMPT_BEAM)
PREFILL_SEED = wl.workload_seed(3)
STOP_ID = 151643


def prefill_flops(lengths, n_q_heads, head_dim) -> float:
    L = np.asarray(lengths, dtype=np.float64)
    return float(np.sum(4.0 * head_dim * L * (L + 1) / 2.0) * n_q_heads)


def prefill_bytes(T, n_q_heads, n_kv_heads, head_dim) -> float:
    # read Q, K, V once, write O once (bf16)
    return float(T) * (2 * n_q_heads + 2 * n_kv_heads) * head_dim * 2


def select_bytes(W_in, V) -> float:
    return float(W_in) * V * 2


def select_launches(W_in, V, W) -> int:
    """Kernels one slm_beam_select call launches: stream + select when the
    group keys fit the select kernel's shared memory (rows of at most 64 tiles
    of 8192 logits, at most 16,384 groups: tiles when there are at least 2W of
    them, else their 128 sub-chunks each), else a row-statistics kernel too."""
    n_tpr = -(-V // 8192)
    n_tiles = W_in * n_tpr
    n_groups = n_tiles if n_tiles >= 2 * W else n_tiles * 128
    return 2 if (n_tpr <= 64 and n_groups <= 16384) else 3


def decode_attn_bytes(W, Lp, L_prev, Hq, Hkv, D) -> float:
    row = Hkv * D * 2
    q_o = 2 * W * Hq * D * 2
    prefix = 2 * Lp * row
    suffix_read = 2 * W * L_prev * row + 2 * W * row  # parents' history + new rows
    suffix_write = 2 * W * (L_prev + 1) * row
    return float(q_o + prefix + suffix_read + suffix_write)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling every 50 ms on a reader thread; summary() keeps the
    samples taken between mark_start() and mark_end() (the timed region)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []  # (host time, line)
        self.t0 = self.t1 = None
        self.thread = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        deadline = time.perf_counter() + 5.0  # sampling must be running before the timed region
        while not self.lines and time.perf_counter() < deadline:
            time.sleep(0.01)
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        t0 = self.t0 if self.t0 is not None else -1e30
        t1 = (self.t1 if self.t1 is not None else 1e30) + 0.05
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock sample inside the timed region"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# DRAM bytes (read + write) per prefill launch on this workload, from an ncu
# capture of `bench.py --ncu-case prefill` (one layer of the same batch), keyed
# by the code it was taken on (the kernel, its PTX helpers and the host launch,
# comments and blank space left out); any other code reports null.
PREFILL_TRAFFIC = {"12fba8de95f366fe": 1.199149e9 + 0.512910e9}


def prefill_code_key() -> str:
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("attn_fwd.cuh", "sm103_ptx.cuh", "api.cu"):
        with open(os.path.join(ROOT, "attention_packed_varlen_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def prefill_traffic():
    try:
        return PREFILL_TRAFFIC.get(prefill_code_key())
    except OSError:
        return None


# ----------------------------------------------------------------------------
# Synthetic inputs on the device
# ----------------------------------------------------------------------------
def device_randn(shape, gen, dev, std=1.0):
    x = torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


class PrefillSet:
    def __init__(self, dev, layers: int, seed: int):
        w = PREFILL_WL
        self.lengths = wl.draw_lengths(w.n_seqs, w.len_lo, w.len_hi, seed)
        self.T = int(self.lengths.sum())
        self.max_seqlen = int(self.lengths.max())
        self.cu_host = wl.cu_seqlens_from_lengths(self.lengths)
        self.cu = self.cu_host.to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        self.layers = []
        for _ in range(layers):
            q = device_randn((self.T, w.n_q_heads, w.head_dim), gen, dev)
            k = device_randn((self.T, w.n_kv_heads, w.head_dim), gen, dev)
            v = device_randn((self.T, w.n_kv_heads, w.head_dim), gen, dev)
            self.layers.append((q, k, v, torch.empty_like(q)))
        from attention_packed_varlen_gb300 import _binding as slm
        need = slm.slm_prefill_workspace_size(w.n_seqs, self.T, self.max_seqlen, w.n_q_heads, w.n_kv_heads)
        self.ws = torch.empty(need, dtype=torch.uint8, device=dev)
        self.flops = prefill_flops(self.lengths, w.n_q_heads, w.head_dim)
        self.bytes = prefill_bytes(self.T, w.n_q_heads, w.n_kv_heads, w.head_dim)


class BeamSet:
    def __init__(self, dev, bw: wl.BeamWorkload, seed: int):
        self.w = bw
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        W, Hq, Hkv, D, S = bw.beams, bw.n_q_heads, bw.n_kv_heads, bw.head_dim, bw.max_suffix
        self.kp = device_randn((bw.prefix_len, Hkv, D), gen, dev)
        self.vp = device_randn((bw.prefix_len, Hkv, D), gen, dev)
        self.ks = [torch.zeros((W, S, Hkv, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.vs = [torch.zeros((W, S, Hkv, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.steps = []
        rng = np.random.default_rng(seed)
        for _ in range(bw.steps):
            q = device_randn((W, Hq, D), gen, dev)
            kn = device_randn((W, Hkv, D), gen, dev)
            vn = device_randn((W, Hkv, D), gen, dev)
            parent = torch.from_numpy(rng.integers(0, W, W).astype(np.int32)).to(dev)
            logits = device_randn((W, bw.vocab), gen, dev, std=bw.logit_std)
            self.steps.append((q, kn, vn, parent, logits))
        self.cum = torch.zeros(W, dtype=torch.float32, device=dev)
        self.o = torch.empty((W, Hq, D), dtype=torch.bfloat16, device=dev)
        from attention_packed_varlen_gb300 import _binding as slm
        self.ws = torch.empty(slm.slm_beam_select_workspace_size(W, bw.vocab, W), dtype=torch.uint8, device=dev)
        dws = slm.slm_shared_prefix_decode_workspace_size(W, bw.prefix_len, Hq, Hkv, D)
        self.dec_ws = torch.zeros(max(dws, 1), dtype=torch.uint8, device=dev)
        self.res = {
            "token": torch.empty(W, dtype=torch.int32, device=dev),
            "parent": torch.empty(W, dtype=torch.int32, device=dev),
            "score": torch.empty(W, dtype=torch.float32, device=dev),
            "cand_token": torch.empty(2 * W, dtype=torch.int32, device=dev),
            "cand_parent": torch.empty(2 * W, dtype=torch.int32, device=dev),
            "cand_score": torch.empty(2 * W, dtype=torch.float32, device=dev),
        }


def run_prefill_layer(slm_lib, ps: PrefillSet, layer, stream_ptr):
    import ctypes
    w = PREFILL_WL
    q, k, v, o = layer
    st = slm_lib.slm_packed_prefill_attn(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(ps.cu.data_ptr()), None, w.n_seqs, ps.T, ps.max_seqlen, w.n_q_heads, w.n_kv_heads,
        w.head_dim, w.softmax_scale, ctypes.c_void_p(o.data_ptr()), None, ctypes.c_void_p(ps.ws.data_ptr()),
        ps.ws.numel(), None, stream_ptr)
    if st != 0:
        raise RuntimeError(slm_lib.slm_last_error().decode())


def run_decode_step(slm_lib, bs: BeamSet, t: int, stream_ptr):
    import ctypes
    bw = bs.w
    q, kn, vn, parent, logits = bs.steps[t]
    ks_in, vs_in = bs.ks[t % 2], bs.vs[t % 2]
    ks_out, vs_out = bs.ks[(t + 1) % 2], bs.vs[(t + 1) % 2]
    P = lambda x: ctypes.c_void_p(x.data_ptr())
    st = slm_lib.slm_shared_prefix_decode_attn(
        P(q), P(bs.kp), P(bs.vp), P(ks_in), P(vs_in), P(kn), P(vn), P(parent), bw.beams, bw.prefix_len, t,
        bw.max_suffix, bw.n_q_heads, bw.n_kv_heads, bw.head_dim, bw.softmax_scale, P(ks_out), P(vs_out), P(bs.o),
        None, None, P(bs.dec_ws), bs.dec_ws.numel(), stream_ptr)
    if st != 0:
        raise RuntimeError(slm_lib.slm_last_error().decode())
    run_select(slm_lib, bs, t, stream_ptr)


def run_select(slm_lib, bs: BeamSet, t: int, stream_ptr):
    """The step's beam selection over its fresh logits [W, V]."""
    import ctypes
    bw = bs.w
    logits = bs.steps[t][4]
    P = lambda x: ctypes.c_void_p(x.data_ptr())
    r = bs.res
    st = slm_lib.slm_beam_select(
        P(logits), P(bs.cum), bw.beams, bw.vocab, bw.beams, P(r["token"]), P(r["parent"]), P(r["score"]),
        P(r["cand_token"]), P(r["cand_parent"]), P(r["cand_score"]), None, P(bs.ws), bs.ws.numel(), stream_ptr)
    if st != 0:
        raise RuntimeError(slm_lib.slm_last_error().decode())


def loop_bytes(bw) -> float:
    """Algorithmic bytes of one fixed-depth loop: the first step's one logits
    row, then per decode step the attention's bytes and the step's logits."""
    b = select_bytes(1, bw.vocab)
    for t in range(1, bw.steps + 1):
        b += decode_attn_bytes(bw.beams, bw.prefix_len, t - 1, bw.n_q_heads, bw.n_kv_heads, bw.head_dim)
        b += select_bytes(bw.beams, bw.vocab)
    return float(b)


class L2Flush:
    """Writes a buffer twice the size of L2 between timed repetitions."""

    def __init__(self, dev, nbytes: int = 256 << 20):
        self.buf = torch.empty(nbytes // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.buf.zero_()


def timed_reps(fn, stream, reps: int, warmup: int, flush=None):
    """Median CUDA-event time (s) of fn() on `stream`, L2 flushed before each rep."""
    for _ in range(warmup):
        fn()
    ms = []
    for _ in range(reps):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms) / 1e3


def measure_decode_loop(dev, bw, seed, stop_id, stream, peaks, flush, reps=20, warmup=3):
    """The fixed-depth loop (first step + bw.steps decode steps) captured as
    one CUDA graph: replay time, and the same loop enqueued call by call."""
    from attention_packed_varlen_gb300.decode_loop import BeamDecodeLoop
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    W, Hq, Hkv, D, V = bw.beams, bw.n_q_heads, bw.n_kv_heads, bw.head_dim, bw.vocab
    logits0 = device_randn((1, V), gen, dev, std=bw.logit_std)
    kp = device_randn((bw.prefix_len, Hkv, D), gen, dev)
    vp = device_randn((bw.prefix_len, Hkv, D), gen, dev)
    steps = [(device_randn((W, Hq, D), gen, dev), device_randn((W, Hkv, D), gen, dev),
              device_randn((W, Hkv, D), gen, dev), device_randn((W, V), gen, dev, std=bw.logit_std))
             for _ in range(bw.steps)]
    if stop_id is not None:  # a third of the rows rank the stop token first
        for st in steps:
            rows = torch.arange(0, W, 3, device=dev)
            st[3][rows, stop_id] = (st[3][rows].float().amax(dim=1) + 0.5).to(torch.bfloat16)
    loop = BeamDecodeLoop(W, V, bw.steps, bw.prefix_len, Hq, Hkv, D, stop_id=stop_id,
                          softmax_scale=bw.softmax_scale, device=dev)
    loop.capture(logits0, kp, vp, steps)
    graph_s = timed_reps(loop.replay, stream, reps, warmup, flush)
    eager_s = timed_reps(lambda: loop.record(logits0, kp, vp, steps), stream, reps, warmup, flush)
    from attention_packed_varlen_gb300 import _binding as slm
    slm.slm_check_status(loop.status)
    n = bw.steps
    launches = (select_launches(1, V, W) + 1 + n * (1 + select_launches(W, V, W) + 1)
                + ((n + 1) if stop_id is not None else 0))
    nbytes = loop_bytes(bw)
    return {"stop_id": stop_id, "decode_steps": n, "graph_us_per_loop": graph_s * 1e6,
            "graph_us_per_decode_step": graph_s * 1e6 / n, "eager_us_per_loop": eager_s * 1e6,
            "launches_per_loop": launches, "bytes_per_loop": nbytes,
            "hbm_frac_of_measured": nbytes / graph_s / 1e9 / peaks["hbm_gbs"]}


def measure_prefill_configs(dev, stream, peaks, flush, reps=50, warmup=10):
    """The tiny packed prefill and the one-layer Prefill-Only request: median
    of `reps` replays of the call (schedule + attention) captured in a CUDA
    graph, cold (L2 flushed before each replay) and hot (the same inputs
    again, L2 warm); the graph keeps host launch time out of both."""
    from attention_packed_varlen_gb300 import _binding as slm
    out = {}
    for w, seed in ((wl.TINY_PREFILL, wl.workload_seed(1)), (wl.PREFILL_ONLY_REQUEST, wl.workload_seed(2))):
        lengths = wl.draw_lengths(w.n_seqs, w.len_lo, w.len_hi, seed) if w.lengths is None else np.asarray(w.lengths)
        T = int(lengths.sum())
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        q = device_randn((T, w.n_q_heads, w.head_dim), gen, dev)
        k = device_randn((T, w.n_kv_heads, w.head_dim), gen, dev)
        v = device_randn((T, w.n_kv_heads, w.head_dim), gen, dev)
        cu = wl.cu_seqlens_from_lengths(lengths).to(dev)
        o = torch.empty_like(q)
        ws = torch.empty(slm.slm_prefill_workspace_size(len(lengths), T, int(lengths.max()), w.n_q_heads,
                                                        w.n_kv_heads), dtype=torch.uint8, device=dev)
        call = lambda: slm.slm_packed_prefill_attn(q, k, v, cu, int(lengths.max()), w.softmax_scale, out=o,
                                                   workspace=ws)
        call()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        fn = graph.replay
        flops = prefill_flops(lengths, w.n_q_heads, w.head_dim)
        nbytes = prefill_bytes(T, w.n_q_heads, w.n_kv_heads, w.head_dim)
        t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        res = {"tokens": T, "gflop": flops / 1e9, "mbytes": nbytes / 1e6,
               "roofline_floor_us": max(t_tensor, t_hbm) * 1e6,
               "bound": "hbm" if t_hbm > t_tensor else "tensor"}
        for kind, fl in (("cold", flush), ("hot", None)):
            t = timed_reps(fn, stream, reps, warmup, fl)
            res[kind] = {"us": t * 1e6, "tflops": flops / t / 1e12,
                         "frac_of_bf16_burst": flops / t / 1e12 / peaks["bf16_tflops"],
                         "frac_of_roofline_floor": max(t_tensor, t_hbm) / t,
                         "hbm_gbs": nbytes / t / 1e9}
        out[w.name] = res
    return out


def measure_decode_batched(dev, stream, peaks, flush, reps=20, warmup=3, R=16):
    """R requests' decode attention (the last step of each beam workload:
    longest suffix) back to back in one CUDA graph: sustained GB/s of the
    attention alone, L2 flushed before each replay."""
    from attention_packed_varlen_gb300 import _binding as slm
    out = {}
    for bw in BEAM_WLS:
        W, Hq, Hkv, D, S = bw.beams, bw.n_q_heads, bw.n_kv_heads, bw.head_dim, bw.max_suffix
        L_prev = bw.steps - 1
        gen = torch.Generator(device=dev)
        gen.manual_seed(rank_beam_seed(bw, 0) + 31)
        reqs = []
        for _ in range(R):
            reqs.append(dict(
                q=device_randn((W, Hq, D), gen, dev), kp=device_randn((bw.prefix_len, Hkv, D), gen, dev),
                vp=device_randn((bw.prefix_len, Hkv, D), gen, dev), ks=device_randn((W, S, Hkv, D), gen, dev),
                vs=device_randn((W, S, Hkv, D), gen, dev), kn=device_randn((W, Hkv, D), gen, dev),
                vn=device_randn((W, Hkv, D), gen, dev),
                parent=torch.randint(0, W, (W,), generator=gen, device=dev, dtype=torch.int32),
                ks_out=torch.empty((W, S, Hkv, D), dtype=torch.bfloat16, device=dev),
                vs_out=torch.empty((W, S, Hkv, D), dtype=torch.bfloat16, device=dev),
                o=torch.empty((W, Hq, D), dtype=torch.bfloat16, device=dev)))
        n = slm.slm_shared_prefix_decode_workspace_size(W, bw.prefix_len, Hq, Hkv, D)
        ws = torch.zeros(max(n, 16), dtype=torch.uint8, device=dev)

        def all_calls():
            for r in reqs:
                slm.slm_shared_prefix_decode_attn(r["q"], r["kp"], r["vp"], r["ks"], r["vs"], r["kn"], r["vn"],
                                                  r["parent"], L_prev, bw.softmax_scale, ks_out=r["ks_out"],
                                                  vs_out=r["vs_out"], out=r["o"], workspace=ws if n else None)
        all_calls()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            all_calls()
        t = timed_reps(g.replay, stream, reps, warmup, flush)
        nbytes = R * decode_attn_bytes(W, bw.prefix_len, L_prev, Hq, Hkv, D)
        out[bw.name] = {"requests": R, "us_per_call": t * 1e6 / R, "bytes_per_call": nbytes / R,
                        "sustained_gbs": nbytes / t / 1e9, "hbm_frac_of_measured": nbytes / t / 1e9 / peaks["hbm_gbs"],
                        "l2": "flushed before each graph replay"}
    return out


def measure_heads(dev, stream, peaks, flush, T, reps=20, warmup=3):
    """Fused SwiGLU + per-token E4M3 over the concurrent batch's token rows
    (intermediate 5632), and last-token label scores of its 240 sequences."""
    from attention_packed_varlen_gb300 import _binding as slm
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.workload_seed(6))
    I = 5632
    gu = device_randn((T, 2 * I), gen, dev, std=2.0)
    s = timed_reps(lambda: slm.slm_swiglu_quant_e4m3(gu), stream, reps, warmup)
    nbytes = float(T) * (2 * I * 2 + I + 4)
    swiglu = {"tokens": T, "intermediate": I, "us": s * 1e6, "bytes": nbytes,
              "achieved_gbs": nbytes / s / 1e9, "hbm_frac_of_measured": nbytes / s / 1e9 / peaks["hbm_gbs"],
              "l2": "input 2x larger than L2 per call"}
    del gu
    lengths = wl.draw_lengths(PREFILL_WL.n_seqs, PREFILL_WL.len_lo, PREFILL_WL.len_hi, PREFILL_SEED)
    cu = wl.cu_seqlens_from_lengths(lengths).to(dev)
    d_model, n_labels = 2048, 8
    hidden = device_randn((int(lengths.sum()), d_model), gen, dev)
    w_label = device_randn((n_labels, d_model), gen, dev, std=0.05)
    s = timed_reps(lambda: slm.slm_label_scores(hidden, cu, w_label), stream, reps, warmup, flush)
    labels = {"sequences": len(lengths), "d_model": d_model, "n_labels": n_labels, "us": s * 1e6,
              "bytes": float(len(lengths) * d_model * 2 + n_labels * d_model * 2),
              "l2": "flushed before each call"}
    return {"swiglu_e4m3": swiglu, "label_scores": labels}


# ----------------------------------------------------------------------------
# CPU oracle timing (bounded sample)
# ----------------------------------------------------------------------------
def oracle_prefill_sample(budget_s: float = 15.0):
    """Times the fp64 C oracle on whole sequences of the same batch (all host
    cores), adding sequences until about budget_s of work.  Returns
    (TFLOP/s, cores, description)."""
    import oracle
    w = PREFILL_WL
    lengths = wl.draw_lengths(w.n_seqs, w.len_lo, w.len_hi, PREFILL_SEED)
    cores = oracle.default_threads()
    done_flops, elapsed, n_seq = 0.0, 0.0, 0
    # sequences in order; each is an independent causal problem
    for b, L in enumerate(lengths):
        if elapsed >= budget_s:
            break
        inp = wl.prefill_inputs([int(L)], w.n_q_heads, w.n_kv_heads, w.head_dim, seed=PREFILL_SEED * 1000 + b)
        t0 = time.perf_counter()
        oracle.packed_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens.numpy(), inp.softmax_scale, n_threads=cores)
        elapsed += time.perf_counter() - t0
        done_flops += prefill_flops([int(L)], w.n_q_heads, w.head_dim)
        n_seq += 1
    tflops = done_flops / elapsed / 1e12
    desc = (f"fp64 C oracle (OpenMP over rows) on {n_seq} of the batch's {w.n_seqs} sequences "
            f"({done_flops / 1e9:.1f} GFLOP of the layer's {prefill_flops(lengths, w.n_q_heads, w.head_dim) / 1e9:.0f}), "
            f"{elapsed:.1f} s")
    return tflops, cores, desc


def oracle_timings(budget_s: float = 8.0):
    """The oracle as it stands on the host cores, single-threaded and on all
    cores: prefill on whole sequences of the concurrent batch (about
    budget_s each), one decode step of the long-prompt wide beam (W = 400,
    4 history rows), and one beam selection of the short-prompt beam (a full
    sort of 100 x 151,936 candidates; the sort is single-threaded)."""
    import oracle
    w = PREFILL_WL
    lengths = wl.draw_lengths(w.n_seqs, w.len_lo, w.len_hi, PREFILL_SEED)
    cores = oracle.default_threads()
    res = {"cores": cores, "cpu": cpu_model()}
    for threads in (1, cores):
        done, elapsed, n_seq = 0.0, 0.0, 0
        for b, L in enumerate(lengths):
            if elapsed >= budget_s:
                break
            inp = wl.prefill_inputs([int(L)], w.n_q_heads, w.n_kv_heads, w.head_dim, seed=PREFILL_SEED * 1000 + b)
            t0 = time.perf_counter()
            oracle.packed_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens.numpy(), inp.softmax_scale, n_threads=threads)
            elapsed += time.perf_counter() - t0
            done += prefill_flops([int(L)], w.n_q_heads, w.head_dim)
            n_seq += 1
        res[f"prefill_{threads}_threads"] = {"tflops": done / elapsed / 1e12, "sequences": n_seq, "s": elapsed}
    bw = wl.LONG_PROMPT_WIDE_BEAM
    d = wl.decode_inputs(bw.beams, bw.prefix_len, bw.steps - 1, bw.max_suffix, bw.n_q_heads, bw.n_kv_heads,
                         bw.head_dim, seed=wl.workload_seed(5, bw.steps - 1))
    for threads in (1, cores):
        t0 = time.perf_counter()
        oracle.shared_prefix_decode(d.q, d.kp, d.vp, d.ks, d.vs, d.k_new, d.v_new, d.parent, d.L_prev,
                                    d.softmax_scale, n_threads=threads)
        res[f"decode_attention_{threads}_threads"] = {"us_per_step": (time.perf_counter() - t0) * 1e6,
                                                       "workload": bw.name}
    bs = wl.SHORT_PROMPT_BEAM
    s = wl.select_inputs(bs.beams, bs.vocab, bs.beams, seed=wl.workload_seed(4, 1), step=1)
    t0 = time.perf_counter()
    oracle.beam_select(s.logits, s.cum, 2 * bs.beams)
    res["beam_select_1_thread"] = {"us_per_step": (time.perf_counter() - t0) * 1e6, "workload": bs.name}
    return res


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


# ----------------------------------------------------------------------------
# Arms
# ----------------------------------------------------------------------------
def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        torch.distributed.init_process_group(backend=backend)
    return rank, world, local


def rank_prefill_seed(rank: int) -> int:
    """Each rank draws its own independent batch of the same workload (weak
    scaling: the units are whole requests, nothing is exchanged)."""
    return PREFILL_SEED + 7919 * rank


def rank_beam_seed(bw, rank: int) -> int:
    return wl.workload_seed(5 if bw is wl.LONG_PROMPT_WIDE_BEAM else 4) + rank


def max_over_ranks_of(x: float, world: int, dev) -> float:
    """The slowest rank's time: the job is done when every rank is."""
    if world == 1:
        return x
    tt = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(units_per_rank: float, world: int, slowest_s: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return units_per_rank * world / slowest_s


def run_reference(args):
    rank, world, _ = dist_setup(args)
    if rank != 0:
        return
    steps = []
    tfl, cores, desc = None, None, None
    for _ in range(args.warmup + args.steps):
        tfl, cores, desc = oracle_prefill_sample(budget_s=args.ref_budget)
        steps.append(tfl)
    timed = steps[args.warmup:]
    value = float(np.median(timed))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL_WL.name, "layers_timed": "bounded sample of one layer"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gpu(args):
    rank, world, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from attention_packed_varlen_gb300 import _binding as slm
    lib = slm.load()
    peaks = load_peaks()
    seed = rank_prefill_seed(rank)

    ps = PrefillSet(dev, PREFILL_WL.layers, seed)
    beams = [BeamSet(dev, bw, rank_beam_seed(bw, rank)) for bw in BEAM_WLS]
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    import ctypes
    sp = ctypes.c_void_p(stream.cuda_stream)
    n_pre = len(ps.layers)
    n_dec = [bs.w.steps for bs in beams]

    def one_step(rec=None):
        for i, layer in enumerate(ps.layers):
            if rec is not None:
                rec["pre"][i][0].record(stream)
            run_prefill_layer(lib, ps, layer, sp)
            if rec is not None:
                rec["pre"][i][1].record(stream)
        for j, bs in enumerate(beams):
            for t in range(bs.w.steps):
                if rec is not None:
                    rec["dec"][j][t][0].record(stream)
                run_decode_step(lib, bs, t, sp)
                if rec is not None:
                    rec["dec"][j][t][1].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    recs = [{"pre": [mk() for _ in range(n_pre)], "dec": [[mk() for _ in range(n)] for n in n_dec]}
            for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        t_start.record(stream)
        for k in range(args.steps):
            one_step(recs[k])
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [s.elapsed_time(e) for r in recs for (s, e) in r["pre"]]
    dec_ms = [[[r["dec"][j][t][0].elapsed_time(r["dec"][j][t][1]) for t in range(n_dec[j])] for r in recs]
              for j in range(len(beams))]

    max_over_ranks = lambda x: max_over_ranks_of(x, world, dev)
    prefill_time_s = max_over_ranks(sum(pre_ms) / 1e3)
    total_ms = max_over_ranks(total_ms)
    value = job_throughput(ps.flops * n_pre * args.steps, world, prefill_time_s) / 1e12
    avg_launch_s = sum(pre_ms) / len(pre_ms) / 1e3
    achieved = ps.flops / avg_launch_s / 1e12

    decode = {}
    for j, bs in enumerate(beams):
        bw = bs.w
        per_step_us = max_over_ranks(float(np.mean(dec_ms[j]))) * 1e3
        bytes_step = np.mean([decode_attn_bytes(bw.beams, bw.prefix_len, t, bw.n_q_heads, bw.n_kv_heads,
                                                bw.head_dim) for t in range(bw.steps)])
        bytes_step += select_bytes(bw.beams, bw.vocab)
        decode[bw.name] = {"us_per_step": per_step_us, "bytes_per_step": float(bytes_step),
                           "hbm_frac_of_measured": float(bytes_step / (per_step_us * 1e-6) / 1e9 / peaks["hbm_gbs"])}

    # e2e: the same prefill metric through the public API from pinned host
    # buffers: per layer, copy Q/K/V in, run, copy O out (one layer's host set
    # reused for every layer).  Copies in, attention and copies out run on
    # three streams over two device buffer sets, so layer i+1's inputs arrive
    # and layer i-1's output leaves while layer i computes.
    e2e = None
    if args.e2e_layers > 0:
        q0, k0, v0, _ = ps.layers[0]
        hq = torch.empty(q0.shape, dtype=q0.dtype, pin_memory=True)
        hk = torch.empty(k0.shape, dtype=k0.dtype, pin_memory=True)
        hv = torch.empty(v0.shape, dtype=v0.dtype, pin_memory=True)
        ho = torch.empty(q0.shape, dtype=q0.dtype, pin_memory=True)
        hq.copy_(q0)
        hk.copy_(k0)
        hv.copy_(v0)
        bufs = [(torch.empty_like(q0), torch.empty_like(k0), torch.empty_like(v0), torch.empty_like(q0))
                for _ in range(2)]
        s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        sp_run = ctypes.c_void_p(s_run.cuda_stream)
        ev = lambda: torch.cuda.Event()
        loaded, ran, stored = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s_ in (s_in, s_run, s_out):
            s_.wait_event(e0)
        for i in range(args.e2e_layers):
            b = i % 2
            dq, dk, dv, do = bufs[b]
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(ran[b])        # layer i-2 has read this set
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                loaded[b].record(s_in)
            s_run.wait_event(loaded[b])
            if used[b]:
                s_run.wait_event(stored[b])        # layer i-2's output has left
            run_prefill_layer(lib, ps, (dq, dk, dv, do), sp_run)
            ran[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ran[b])
                ho.copy_(do, non_blocking=True)
                stored[b].record(s_out)
            used[b] = True
        for s_ in (s_in, s_run, s_out):
            stream.wait_stream(s_)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3)
        h2d = (hq.numel() + hk.numel() + hv.numel()) * 2 * args.e2e_layers
        d2h = ho.numel() * 2 * args.e2e_layers
        e2e = {"value": job_throughput(ps.flops * args.e2e_layers, world, e2e_s) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "layers": args.e2e_layers,
               # the copies overlap the attention: the link, not the kernel, bounds this figure
               "h2d_gbs": h2d / e2e_s / 1e9, "d2h_gbs": d2h / e2e_s / 1e9}

    # the fused fixed-depth loop (one CUDA graph) and the head kernels, timed
    # after the main step with their own events
    flush = L2Flush(dev)
    decode_loop = {}
    heads = None
    prefill_cfgs = decode_batched = None
    if not args.no_extra_legs:
        prefill_cfgs = measure_prefill_configs(dev, stream, peaks, flush)
        decode_batched = measure_decode_batched(dev, stream, peaks, flush)
        for j, bs in enumerate(beams):
            bw = bs.w
            decode_loop[bw.name] = {
                "plain": measure_decode_loop(dev, bw, rank_beam_seed(bw, rank) + 1, None, stream, peaks, flush),
                "with_stop_token": measure_decode_loop(dev, bw, rank_beam_seed(bw, rank) + 2, STOP_ID, stream,
                                                       peaks, flush)}
        heads = measure_heads(dev, stream, peaks, flush, ps.T)

    cpu = None
    oracle_t = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tfl, cores, desc = oracle_prefill_sample(budget_s=args.ref_budget)
        cpu = {"value": tfl, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "cpu": cpu_model()}
        if not args.no_extra_legs:
            oracle_t = oracle_timings()

    # prefill: schedule + attention; decode step: attention + the selection's kernels
    launches_per_step = n_pre * 2 + sum(n_dec[j] * (1 + select_launches(b.w.beams, b.w.vocab, b.w.beams))
                                        for j, b in enumerate(beams))
    peak_sust = peaks["bf16_tflops_sustained"]
    peak_burst = peaks["bf16_tflops"]
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": PREFILL_WL.name + " + beam decode steps (" + "; ".join(b.name for b in BEAM_WLS) + ")",
            "prefill_tokens_per_layer": ps.T, "prefill_layers": n_pre,
            "prefill_gflop_per_layer": ps.flops / 1e9,
            "l2": "inputs larger than L2: 28 distinct 1.6 GB layer sets per step",
            "parallelism": f"replicas x{world}",
        },
        "prefill_pct_of_bf16_peak": {"burst": value / world / peak_burst, "sustained": value / world / peak_sust,
                                     "sm_mhz": clocks.get("sm_mhz")},
        "decode": decode,
        "decode_batched_graph": decode_batched,
        "prefill_configs": prefill_cfgs,
        "decode_loop_graph": decode_loop,
        "heads": heads,
        # the prefill runs at the maximum SM clock through the step (see
        # clocks), so the burst peak is its denominator; the sustained one,
        # measured at a lower clock under the power cap, is given beside it
        "roofline": {"kernel": "slm_packed_prefill_attn (schedule + tcgen05 attention)", "bound": "tensor",
                     "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s", "frac": achieved / peak_burst,
                     "peak_kind": f"bf16 burst, {peaks['source']}",
                     "frac_of_sustained": achieved / peak_sust, "sm_mhz": clocks.get("sm_mhz"),
                     "hbm_achieved_gbs": ps.bytes / avg_launch_s / 1e9,
                     "hbm_frac": ps.bytes / avg_launch_s / 1e9 / peaks["hbm_gbs"],
                     "traffic": args.traffic if args.traffic is not None else prefill_traffic()},
        "clocks": clocks,
        "oracle_timings": oracle_t,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_ncu_case(args):
    """One kernel on a reduced input for an ncu capture (a few hundred MB to
    ~1 GB on the device, still larger than L2), three calls so a capture can
    skip the first two."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from attention_packed_varlen_gb300 import _binding as slm
    lib = slm.load()
    import ctypes
    sp = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    if args.ncu_case == "prefill":
        ps = PrefillSet(dev, 1, PREFILL_SEED)   # one layer of the 240-sequence batch (1.6 GB)
        for _ in range(3):
            run_prefill_layer(lib, ps, ps.layers[0], sp)
    elif args.ncu_case == "select":  # stream + select of the W=400 selection (121.5 MB of logits)
        bw = wl.LONG_PROMPT_WIDE_BEAM
        bs = BeamSet(dev, bw, wl.workload_seed(5))
        for _ in range(3):
            run_select(lib, bs, bw.steps - 1, sp)
    else:
        bw = wl.LONG_PROMPT_WIDE_BEAM
        bs = BeamSet(dev, bw, wl.workload_seed(5))
        for _ in range(3):
            run_decode_step(lib, bs, bw.steps - 1, sp)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": args.ncu_case, "ok": True}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-layers", type=int, default=28)
    ap.add_argument("--ref-budget", type=float, default=15.0, help="seconds of oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-legs", action="store_true",
                    help="skip the decode-loop graph and head-kernel timings")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per prefill launch from an ncu capture of the current kernel")
    ap.add_argument("--ncu-case", choices=["prefill", "decode", "select"], default=None,
                    help="run one kernel on a reduced input for an ncu capture, then exit")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
