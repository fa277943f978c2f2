"""Benchmark of the rotated 4-bit KV-cache decode path on GB300.

Workload (default): full decode step at 256k context -- 8 sequences at 262,144 cached
positions over a 50-layer stack (every fifth layer full attention with the rotated int4
cache, the other 40 sliding-window layers with window 513 and an FP8 e4m3 cache), 20
query / 4 KV heads of 128, bf16 inputs, one query row per sequence, timed over K
consecutive decode steps (each step appends one token per sequence and layer). Inputs
are seeded synthetic data (synth) already resident in HBM; the int4 cache alone is
11.4 GB, far larger than L2, so no flush is needed between steps.

Prints one JSON line: session-steps/s (value), the HBM roofline of the int4 attention
call, the 64k point (32 ragged sequences, one int4 layer), an end-to-end figure with
host<->device copies, and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference]
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "int4 decode-attn HBM GB/s & % of peak; session-steps/s at 64k and 256k context"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- distributed plumbing

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("KVQ_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(ms_local, units_local, world, device="cpu"):
    """Whole-job figure of a weak-scaling run: the slowest rank's time and the units all ranks
    processed divided by it. Returns (ms_max, units_per_second)."""
    ms = max_over_ranks(ms_local, world, device)
    units = units_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(units_local)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        units = float(t.item())
    return ms, units / (ms * 1e-3)


def max_over_ranks(x, world, device="cpu"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- the workload on the GPU

class Stack256k:
    """The 50-layer decode stack with synthetic caches and per-step inputs resident on the device."""

    def __init__(self, steps_total, device, prologue="matrix"):
        import torch

        import synth
        from quantized_kv_cache_fold_gb300.runner import DecodeStack
        from synth.workloads import SWA_K_SCALE, SWA_V_SCALE, config

        w = config(5)
        self.w = w
        self.device = device
        B, S = w.B, 1
        max_pages = w.max_pages(extra_steps=steps_total)
        perm = lambda l, n: synth.page_permutation(w.seed, l, n)  # noqa: E731
        self.st = DecodeStack(B, w.Hq, w.Hkv, S, max_pages, n_layers=w.int4_layers + w.swa_layers, full_every=5,
                              ring_capacity=w.ring_capacity, window=w.window, swa_k_scale=SWA_K_SCALE,
                              swa_v_scale=SWA_V_SCALE, page_perm=perm, device=device)
        st = self.st
        stream = torch.cuda.current_stream().cuda_stream
        from quantized_kv_cache_fold_gb300 import kvq_fp8_append
        for l in st.int4_layers():
            gq, gk = synth.gains(w.seed, l)
            st.set_int4_params(l, synth.rotation_seed(w.seed, l), gq, gk, prologue=prologue)

            def fill(b, p0, T, kb, vb, l=l):
                synth.kv_rows_device(w.seed, l, b, p0, T, w.Hkv, "k", True, kb.data_ptr(), stream)
                synth.kv_rows_device(w.seed, l, b, p0, T, w.Hkv, "v", True, vb.data_ptr(), stream)

            st.prefill_int4(l, w.ctx, fill, chunk_tokens=32768)
        for l in st.swa_layers():
            L = st.layers[l]
            cap = w.ring_capacity
            for b in range(B):
                P = int(w.ctx[b])
                k = torch.empty((cap, w.Hkv, 128), dtype=torch.bfloat16, device=device)
                v = torch.empty_like(k)
                synth.kv_rows_device(w.seed, l, b, P - cap, cap, w.Hkv, "swa_k", True, k.data_ptr(), stream)
                synth.kv_rows_device(w.seed, l, b, P - cap, cap, w.Hkv, "swa_v", True, v.data_ptr(), stream)
                seq = torch.full((cap,), b, dtype=torch.int32, device=device)
                pos = torch.arange(P - cap, P, dtype=torch.int32, device=device)
                kvq_fp8_append(L.ring, k, v, seq, pos, SWA_K_SCALE, SWA_V_SCALE, st.dev_err)
        # per-step inputs: queries and the appended key/value row of every layer
        nL = len(st.layers)
        self.q = torch.empty((steps_total, nL, B, S, w.Hq, 128), dtype=torch.bfloat16, device=device)
        self.kn = torch.empty((steps_total, nL, B, S, w.Hkv, 128), dtype=torch.bfloat16, device=device)
        self.vn = torch.empty_like(self.kn)
        for idx, (buf, sid) in enumerate(((self.q, synth.S_QUERIES), (self.kn, synth.S_KEYS),
                                         (self.vn, synth.S_VALUES))):
            k = synth.key(w.seed + 1000, sid)
            synth.normals_device(k, 0, buf.numel(), buf.data_ptr(), None, True, stream)
        self.ctx = (torch.from_numpy(w.ctx.astype(np.int32)).to(device)[None, :] +
                    torch.arange(steps_total, dtype=torch.int32, device=device)[:, None]).contiguous()
        self.out = torch.empty((nL, B, S, w.Hq, 128), dtype=torch.float32, device=device)
        torch.cuda.synchronize()
        assert st.read_error() == 0, f"device error during set-up: {st.read_error():#x}"
        self.int4 = set(st.int4_layers())
        self.nL = nL

    def step(self, t, ev_pairs=None):
        st = self.st
        for l in range(self.nL):
            if ev_pairs is not None and l in self.int4:
                ev_pairs[0].record()
            st.decode_layer(l, self.q[t, l], self.ctx[t], self.out[l], k_new=self.kn[t, l], v_new=self.vn[t, l])
            if ev_pairs is not None and l in self.int4:
                ev_pairs[1].record()
                ev_pairs = None if len(ev_pairs) == 2 else ev_pairs[2:]

    def int4_call_bytes(self, t):
        """Algorithmic bytes of one int4 layer call at step t: 136 B per token-head over
        ctx + 1 positions of every sequence (K+V codes 128 B, fp16 scale/offset 8 B)."""
        ctx = self.w.ctx + t
        return int((ctx + 1).sum()) * self.w.Hkv * 136

    def launches_per_step(self):
        # int4 layer: prologue/append kernel, split-K attention kernel, combine kernel;
        # window layer: one kernel (append, attention, in-CTA merge)
        return 3 * len(self.int4) + (self.nL - len(self.int4))


# DRAM counters of the int4 attention kernel from one ncu capture on the 64k workload (one
# launch, cold cache): read + write bytes against its algorithmic bytes. The 256k call's traffic
# is that ratio times its own algorithmic bytes (traffic grows with the pages read). The
# counters belong to the kernel sources whose hash is recorded; after any change to them the
# traffic is reported as null until a new capture.
ATTN_CAPTURE = {"dram_read": 906257408, "dram_write": 3086080, "algorithmic": 905157248,
                "sources": ["quantized_kv_cache_fold_gb300/csrc/kvq_attn.cu",
                            "quantized_kv_cache_fold_gb300/csrc/kvq_device.cuh"],
                "sources_sha256_16": "06bd601516a68f61"}


def attn_traffic(call_bytes):
    import hashlib
    hs = hashlib.sha256()
    for f in ATTN_CAPTURE["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            hs.update(fh.read())
    if hs.hexdigest()[:16] != ATTN_CAPTURE["sources_sha256_16"]:
        return None
    c = ATTN_CAPTURE
    return int(round(call_bytes * (c["dram_read"] + c["dram_write"]) / c["algorithmic"]))


def run_64k(device, steps=30, warmup=3):
    """The 64k point: 32 sequences, context U[32768, 65536], one int4 layer, random page order."""
    import torch

    import synth
    from quantized_kv_cache_fold_gb300.runner import DecodeStack
    from synth.workloads import config

    w = config(3)
    perm = lambda l, n: synth.page_permutation(w.seed, l, n)  # noqa: E731
    st = DecodeStack(w.B, w.Hq, w.Hkv, 1, w.max_pages(), 1, 1, page_perm=perm, device=device)
    gq, gk = synth.gains(w.seed, 0)
    st.set_int4_params(0, synth.rotation_seed(w.seed, 0), gq, gk)
    stream = torch.cuda.current_stream().cuda_stream

    def fill(b, p0, T, kb, vb):
        synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "k", True, kb.data_ptr(), stream)
        synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "v", True, vb.data_ptr(), stream)

    st.prefill_int4(0, w.ctx, fill, chunk_tokens=32768)
    q = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.bfloat16, device=device)
    synth.normals_device(synth.key(w.seed + 1000, synth.S_QUERIES), 0, q.numel(), q.data_ptr(), None, True, stream)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).to(device)
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device=device)
    for _ in range(warmup):
        st.decode_layer(0, q, ctx, out)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        e0.record()
        st.decode_layer(0, q, ctx, out)
        e1.record()
    torch.cuda.synchronize()
    assert st.read_error() == 0
    ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    t = statistics.median(ms) * 1e-3
    by = int((w.ctx + 1).sum()) * w.Hkv * 136
    del st
    torch.cuda.empty_cache()
    return {"workload": "32 sequences, context U[32768,65536] (mean %d), one int4 layer, random page order" %
                        int(w.ctx.mean()),
            "int4_call_us": round(t * 1e6, 1), "hbm_gbs": round(by / t / 1e9, 1),
            "session_layer_steps_per_s": round(w.B / t, 1), "algorithmic_bytes": by}


def run_verify(device, steps=30, warmup=3, S_values=(1, 4, 8)):
    """The speculative-verify workload: 64 sequences at 16,384 context, 20/4 heads, S query rows per
    sequence (S = 1, 4, 8) with the S new K/V rows rotated, quantised and appended inside the call
    (at the same positions every repetition), one int4 layer, random page order. Each call is timed
    with CUDA events (median of `steps`); the cache (570 MB) is larger than L2."""
    import torch

    import synth
    from quantized_kv_cache_fold_gb300.runner import DecodeStack
    from synth.workloads import config

    w = config(4)
    peak, _ = measured_peak()
    stream = torch.cuda.current_stream().cuda_stream
    perm = lambda l, n: synth.page_permutation(w.seed, l, n)  # noqa: E731
    Smax = max(S_values)
    st = DecodeStack(w.B, w.Hq, w.Hkv, Smax, w.max_pages() + 1, 1, 1, page_perm=perm, device=device)
    gq, gk = synth.gains(w.seed, 0)
    st.set_int4_params(0, synth.rotation_seed(w.seed, 0), gq, gk)

    def fill(b, p0, T, kb, vb):
        synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "k", True, kb.data_ptr(), stream)
        synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "v", True, vb.data_ptr(), stream)

    st.prefill_int4(0, w.ctx, fill, chunk_tokens=32768)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).to(device)
    rows = []
    for S in S_values:
        q = torch.empty((w.B, S, w.Hq, 128), dtype=torch.bfloat16, device=device)
        kn = torch.empty((w.B, S, w.Hkv, 128), dtype=torch.bfloat16, device=device)
        vn = torch.empty_like(kn)
        for t, key in ((q, synth.S_QUERIES), (kn, synth.S_KEYS), (vn, synth.S_VALUES)):
            synth.normals_device(synth.key(w.seed + 2000 + S, key), 0, t.numel(), t.data_ptr(), None, True, stream)
        out = torch.empty((w.B, S, w.Hq, 128), dtype=torch.float32, device=device)
        for _ in range(warmup):
            st.decode_layer(0, q, ctx, out, k_new=kn, v_new=vn)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(steps, 30))]
        for e0, e1 in evs:
            e0.record()
            st.decode_layer(0, q, ctx, out, k_new=kn, v_new=vn)
            e1.record()
        torch.cuda.synchronize()
        assert st.read_error() == 0
        t = statistics.median([e0.elapsed_time(e1) for e0, e1 in evs]) * 1e-3
        by = int((w.ctx + S).sum()) * w.Hkv * 136
        rows.append({"S": S, "rows_per_kv_head": S * w.G, "int4_call_us": round(t * 1e6, 1),
                     "hbm_gbs": round(by / t / 1e9, 1), "frac_of_measured": round(by / t / 1e9 / peak, 4),
                     "query_rows_per_s": round(w.B * S / t, 1), "algorithmic_bytes": by})
    del st
    torch.cuda.empty_cache()
    return {"workload": "speculative verify: 64 sequences x 16,384 context, 20/4 heads, S new rows appended in "
                        "the call, one int4 layer, random page order", "points": rows}


def run_config2(device, steps=30, warmup=3):
    """16 sequences x 8,192 context, one int4 layer, pages in order, one query row: the cache
    (71 MB) fits in L2, so a 256 MB buffer is written between timed calls (outside the events)
    to flush it."""
    import torch

    import synth
    from quantized_kv_cache_fold_gb300.runner import DecodeStack
    from synth.workloads import config

    w = config(2)
    peak, _ = measured_peak()
    stream = torch.cuda.current_stream().cuda_stream
    st = DecodeStack(w.B, w.Hq, w.Hkv, 1, w.max_pages(), 1, 1, device=device)
    gq, gk = synth.gains(w.seed, 0)
    st.set_int4_params(0, synth.rotation_seed(w.seed, 0), gq, gk)

    def fill(b, p0, T, kb, vb):
        synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "k", True, kb.data_ptr(), stream)
        synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "v", True, vb.data_ptr(), stream)

    st.prefill_int4(0, w.ctx, fill, chunk_tokens=32768)
    q = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.bfloat16, device=device)
    synth.normals_device(synth.key(w.seed + 1000, synth.S_QUERIES), 0, q.numel(), q.data_ptr(), None, True, stream)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).to(device)
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    for _ in range(warmup):
        st.decode_layer(0, q, ctx, out)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (e0, e1) in enumerate(evs):
        flush.fill_(i & 0xFF)
        e0.record()
        st.decode_layer(0, q, ctx, out)
        e1.record()
    torch.cuda.synchronize()
    assert st.read_error() == 0
    t = statistics.median([e0.elapsed_time(e1) for e0, e1 in evs]) * 1e-3
    by = int((w.ctx + 1).sum()) * w.Hkv * 136
    del st, flush
    torch.cuda.empty_cache()
    return {"workload": "16 sequences x 8,192 context, one int4 layer, pages in order, 1 query row",
            "l2": "256 MB buffer written between timed calls", "int4_call_us": round(t * 1e6, 1),
            "hbm_gbs": round(by / t / 1e9, 1), "frac_of_measured": round(by / t / 1e9 / peak, 4),
            "algorithmic_bytes": by}


def run_swa(device, steps=30, warmup=3, sequences=None, layers=None):
    """The 40 FP8 window-513 layers of the 256k step alone (8 sequences x 4 KV heads, 576-slot
    rings, one query row, appended row inside the call), steps captured in one CUDA graph. A
    small case (a few hundred MB) for profiling the window kernel. `sequences` replaces the 8
    sequences by that many, each at the 256k position (the large-batch launch shape); `layers`
    replaces the 40 layers (a smaller device footprint for profiling)."""
    import torch

    import synth
    from quantized_kv_cache_fold_gb300 import kvq_fp8_append, kvq_fp8_swa_plan
    from quantized_kv_cache_fold_gb300.runner import DecodeStack
    from synth.workloads import SWA_K_SCALE, SWA_V_SCALE, config

    w = config(5)
    ctx_all = w.ctx if sequences is None else np.full(sequences, int(w.ctx[0]), np.int64)
    B, S, nL = len(ctx_all), 1, (w.swa_layers if layers is None else layers)
    st = DecodeStack(B, w.Hq, w.Hkv, S, 1, n_layers=nL, full_every=nL + 1, ring_capacity=w.ring_capacity,
                     window=w.window, swa_k_scale=SWA_K_SCALE, swa_v_scale=SWA_V_SCALE, device=device)
    stream = torch.cuda.current_stream().cuda_stream
    cap = w.ring_capacity
    for l in range(nL):
        L = st.layers[l]
        for b in range(B):
            P = int(ctx_all[b])
            k = torch.empty((cap, w.Hkv, 128), dtype=torch.bfloat16, device=device)
            v = torch.empty_like(k)
            synth.kv_rows_device(w.seed, l, b, P - cap, cap, w.Hkv, "swa_k", True, k.data_ptr(), stream)
            synth.kv_rows_device(w.seed, l, b, P - cap, cap, w.Hkv, "swa_v", True, v.data_ptr(), stream)
            seq = torch.full((cap,), b, dtype=torch.int32, device=device)
            pos = torch.arange(P - cap, P, dtype=torch.int32, device=device)
            kvq_fp8_append(L.ring, k, v, seq, pos, SWA_K_SCALE, SWA_V_SCALE, st.dev_err)
    total = warmup + steps
    q = torch.empty((total, nL, B, S, w.Hq, 128), dtype=torch.bfloat16, device=device)
    kn = torch.empty((total, nL, B, S, w.Hkv, 128), dtype=torch.bfloat16, device=device)
    vn = torch.empty_like(kn)
    for buf, sid in ((q, synth.S_QUERIES), (kn, synth.S_KEYS), (vn, synth.S_VALUES)):
        synth.normals_device(synth.key(w.seed + 1000, sid), 0, buf.numel(), buf.data_ptr(), None, True, stream)
    pos0 = (torch.from_numpy(ctx_all.astype(np.int32)).to(device)[None, :] +
            torch.arange(total, dtype=torch.int32, device=device)[:, None]).contiguous()
    out = torch.empty((nL, B, S, w.Hq, 128), dtype=torch.float32, device=device)

    def step(t):
        for l in range(nL):
            st.decode_layer(l, q[t, l], pos0[t], out[l], k_new=kn[t, l], v_new=vn[t, l])

    for t in range(warmup):
        step(t)
    torch.cuda.synchronize()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for i in range(steps):
                step(warmup + i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    assert st.read_error() == 0, f"device error word {st.read_error():#x}"
    us = e0.elapsed_time(e1) * 1e3 / (steps * nL)
    by = int(np.minimum(ctx_all + 1, w.window).sum()) * w.Hkv * 256
    return {"workload": f"{nL} FP8 window-{w.window} layers of the 256k step: {B} sequences x {w.Hkv} KV heads, "
                        f"{cap}-slot rings, 1 query row, appended row in the call",
            "window_layer_us": round(us, 2), "bytes_per_layer": by, "hbm_gbs": round(by / us / 1e3, 1),
            "layers_per_step": nL, "window_us_per_step": round(us * nL, 1),
            "launch_shape": dict(zip(("ctas_per_pair", "streams_per_cta", "stages", "units_per_stream"),
                                     kvq_fp8_swa_plan(cap, B, S, w.Hq, w.Hkv)))}


def run_ab(device, steps=30, warmup=3):
    """A/B of the full-attention formats on the 64k workload (32 sequences, context U[32768,
    65536], one layer, outlier keys): rotated int4 (the method), unrotated int4 (R = I) and FP8
    e4m3 keys and values (the stock format; full attention through the window kernel with the
    window above the context). Per variant: bytes and time per call, and the output's relative L2
    error against exact fp64 attention on unquantised keys and values (torch, sequence 0, all KV
    heads). The FP8 variant's inputs g_k n(k) and g_q n(q) are prepared with torch."""
    import torch

    import synth
    from quantized_kv_cache_fold_gb300 import kvq_fp8_append
    from quantized_kv_cache_fold_gb300.runner import DecodeStack
    from synth.workloads import config

    w = config(3)
    stream = torch.cuda.current_stream().cuda_stream
    gq, gk = synth.gains(w.seed, 0)
    gq_t, gk_t = torch.from_numpy(gq).to(device), torch.from_numpy(gk).to(device)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).to(device)
    q = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.bfloat16, device=device)
    synth.normals_device(synth.key(w.seed + 1000, synth.S_QUERIES), 0, q.numel(), q.data_ptr(), None, True, stream)
    kn = torch.empty((w.B, 1, w.Hkv, 128), dtype=torch.bfloat16, device=device)
    vn = torch.empty_like(kn)
    for b in range(w.B):
        synth.kv_rows_device(w.seed, 0, b, int(w.ctx[b]), 1, w.Hkv, "k", True, kn[b].data_ptr(), stream)
        synth.kv_rows_device(w.seed, 0, b, int(w.ctx[b]), 1, w.Hkv, "v", True, vn[b].data_ptr(), stream)

    def nrm(x):  # n(x) in float32 over the last axis
        x = x.float()
        return x * torch.rsqrt((x * x).mean(dim=-1, keepdim=True) + 1e-6)

    def timed(call):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        ms = []
        for _ in range(steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return statistics.median(ms) * 1e3

    # exact reference for sequence 0: softmax(g_q n(q) . g_k n(k) / sqrt(128)) v over positions 0..ctx0
    L0 = int(w.ctx[0]) + 1
    k0 = torch.empty((L0, w.Hkv, 128), dtype=torch.bfloat16, device=device)
    v0 = torch.empty_like(k0)
    synth.kv_rows_device(w.seed, 0, 0, 0, L0, w.Hkv, "k", True, k0.data_ptr(), stream)
    synth.kv_rows_device(w.seed, 0, 0, 0, L0, w.Hkv, "v", True, v0.data_ptr(), stream)
    kx = (nrm(k0) * gk_t).double()
    qx = (nrm(q[0, 0]) * gq_t).double()
    exact = []
    for h in range(w.Hkv):
        qh = qx[h * w.G:(h + 1) * w.G]
        p = torch.softmax(qh @ kx[:, h].T * 128 ** -0.5, dim=-1)
        exact.append(p @ v0[:, h].double())

    def err_of(out):
        e = []
        for h in range(w.Hkv):
            o = out[0, 0, h * w.G:(h + 1) * w.G].double()
            e.append(((o - exact[h]).norm(dim=-1) / exact[h].norm(dim=-1)).mean().item())
        return float(np.mean(e))

    res = {}
    int4_bytes = int((w.ctx + 1).sum()) * w.Hkv * 136
    for name, rotate in (("int4_rotated", True), ("int4_unrotated", False)):
        perm = lambda l, n: synth.page_permutation(w.seed, 0, n)  # noqa: E731
        st = DecodeStack(w.B, w.Hq, w.Hkv, 1, w.max_pages(), 1, 1, page_perm=perm, device=device)
        st.set_int4_params(0, synth.rotation_seed(w.seed, 0), gq, gk, rotate=rotate)

        def fill(b, p0, T, kb, vb):
            synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "k", True, kb.data_ptr(), stream)
            synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "v", True, vb.data_ptr(), stream)

        st.prefill_int4(0, w.ctx, fill, chunk_tokens=32768)
        out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device=device)
        st.decode_layer(0, q, ctx, out, k_new=kn, v_new=vn)  # the appended row, then time without appends
        torch.cuda.synchronize()
        err = err_of(out)
        us = timed(lambda: st.decode_layer(0, q, ctx, out))
        assert st.read_error() == 0
        res[name] = {"bytes_per_call": int4_bytes, "call_us": round(us, 1),
                     "hbm_gbs": round(int4_bytes / us / 1e3, 1), "rel_l2_err_vs_exact": round(err, 4)}
        del st
        torch.cuda.empty_cache()

    # FP8 keys g_k n(k) and values v for the whole context, per-tensor scales max|x| / 448
    cap = int(-(-(int(w.ctx.max()) + 1) // 64) * 64)
    chunk = 32768
    kbuf = torch.empty((chunk, w.Hkv, 128), dtype=torch.bfloat16, device=device)
    vbuf = torch.empty_like(kbuf)
    kmax = vmax = 0.0
    for b in range(w.B):
        for p0 in range(0, int(w.ctx[b]) + 1, chunk):
            T = min(chunk, int(w.ctx[b]) + 1 - p0)
            synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "k", True, kbuf.data_ptr(), stream)
            synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "v", True, vbuf.data_ptr(), stream)
            kmax = max(kmax, (nrm(kbuf[:T]) * gk_t).abs().max().item())
            vmax = max(vmax, vbuf[:T].float().abs().max().item())
    ks8, vs8 = kmax / 448.0, vmax / 448.0
    st = DecodeStack(w.B, w.Hq, w.Hkv, 1, 1, n_layers=1, full_every=2, ring_capacity=cap, window=cap,
                     swa_k_scale=ks8, swa_v_scale=vs8, device=device)
    ring = st.layers[0].ring
    for b in range(w.B):
        for p0 in range(0, int(w.ctx[b]), chunk):
            T = min(chunk, int(w.ctx[b]) - p0)
            synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "k", True, kbuf.data_ptr(), stream)
            synth.kv_rows_device(w.seed, 0, b, p0, T, w.Hkv, "v", True, vbuf.data_ptr(), stream)
            seq = torch.full((T,), b, dtype=torch.int32, device=device)
            pos = torch.arange(p0, p0 + T, dtype=torch.int32, device=device)
            kvq_fp8_append(ring, (nrm(kbuf[:T]) * gk_t).contiguous(), vbuf[:T].float().contiguous(), seq, pos,
                           ks8, vs8, st.dev_err)
    q8 = (nrm(q) * gq_t).contiguous()
    kn8 = (nrm(kn) * gk_t).contiguous()
    vn8 = vn.float().contiguous()
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device=device)
    st.decode_layer(0, q8, ctx, out, k_new=kn8, v_new=vn8)
    torch.cuda.synchronize()
    err = err_of(out)
    us = timed(lambda: st.decode_layer(0, q8, ctx, out))
    assert st.read_error() == 0
    fp8_bytes = int((w.ctx + 1).sum()) * w.Hkv * 256
    res["fp8"] = {"bytes_per_call": fp8_bytes, "call_us": round(us, 1), "hbm_gbs": round(fp8_bytes / us / 1e3, 1),
                  "rel_l2_err_vs_exact": round(err, 4)}
    del st
    torch.cuda.empty_cache()
    return {"workload": "one full-attention layer, 32 sequences, context U[32768,65536] (mean %d), outlier keys"
                        % int(w.ctx.mean()), "variants": res}


# Kolibri-1's attention stack as the pages describe it: 50 layers, 10 with full attention and
# 40 sliding-window layers (window 513), 4 KV heads of 128.
N_FULL, N_SWA, HKV_MODEL = 10, 40, 4


def session_bytes(fmt: str, ctx_len: int, window_slots: int) -> int:
    """KV bytes one session holds: the 10 full-attention layers at ctx_len positions (int4: 136 B
    per token-head, K and V codes 64 B each plus an fp16 scale and offset each; FP8: 256 B) and the
    40 window layers at window_slots positions of FP8 (256 B per token-head)."""
    per_th = {"int4": 136, "fp8": 256}[fmt]
    return N_FULL * HKV_MODEL * ctx_len * per_th + N_SWA * HKV_MODEL * window_slots * 256


def fill_pool_random(tensors, gen):
    """Seeded random cache contents in place (plumbing: torch's generator; no kernel of the path).
    int4 page blocks: random K and V code bytes (every byte is a valid record), fp16 scales in
    [2^-7, 2^-3) and offsets in (-2, -0.5]; FP8 ring blocks: random e4m3 bytes with the top exponent
    bit cleared (|value| <= 1.875, never NaN)."""
    import torch
    if "pages" in tensors:
        pages = tensors["pages"]
        pages.random_(0, 256, generator=gen)  # in place
        meta = pages[..., 8192:8704].view(torch.int16).unflatten(-1, (128, 2))
        meta[..., 0].random_(0x2000, 0x3000, generator=gen)
        meta[..., 1].random_(-18432, -16384, generator=gen)  # bit patterns 0xB800 .. 0xBFFF
    else:
        data = tensors["data"]
        data.random_(0, 256, generator=gen)
        data.bitwise_and_(0xBF)


def run_capacity(device, budget_gb=160.0, steps=32, warmup=3):
    """Capacity and throughput of a fixed KV pool, rotated int4 full layers against FP8 everywhere.

    A pool of `budget_gb` holds as many sessions as fit at 64k and at 256k context, 50 layers per
    session (10 full-attention layers: int4 pages, 136 B per token-head, or FP8 rings, 256 B; 40
    window-513 layers: 576-slot FP8 rings; session_bytes). The pools hold seeded random codes,
    scales and offsets (fill_pool_random), so scores vary as on data and the attention kernels'
    softmax base moves as it would there. Then the decode step
    (all 50 layers, one query row, the new key/value row appended in each call) is timed for B
    sessions, B from the pool's maximum down to one: each step is one replay of a one-step CUDA
    graph bracketed by events, giving the median step time and the slowest tenth over the median."""
    import torch

    import synth
    from quantized_kv_cache_fold_gb300.runner import DecodeStack
    from synth.workloads import SWA_K_SCALE, SWA_V_SCALE

    Hq, Hkv, G, n_full, n_swa, ring, window = 20, HKV_MODEL, 5, N_FULL, N_SWA, 576, 513
    stream = torch.cuda.current_stream().cuda_stream
    gen = torch.Generator(device=device)
    gen.manual_seed(7)
    result = {"budget_gb": budget_gb, "points": [],
              "fill": "seeded random codes, fp16 scales in [2^-7, 2^-3), offsets in (-2, -0.5]; random e4m3"}
    for ctx_len in (65536, 262144):
        per_session = {fmt: session_bytes(fmt, ctx_len, ring) for fmt in ("int4", "fp8")}
        for fmt in ("int4", "fp8"):
            n_max = int(budget_gb * 1e9 // per_session[fmt])
            max_pages = (ctx_len + 1 + 63) // 64
            cap_full = max_pages * 64
            if fmt == "int4":
                full = DecodeStack(n_max, Hq, Hkv, 1, max_pages, n_layers=n_full, full_every=1, device=device)
                for l in range(n_full):
                    gq, gk = synth.gains(7, l)
                    full.set_int4_params(l, synth.rotation_seed(7, l), gq, gk)
            else:
                full = DecodeStack(n_max, Hq, Hkv, 1, 1, n_layers=n_full, full_every=n_full + 1,
                                   ring_capacity=cap_full, window=cap_full, swa_k_scale=SWA_K_SCALE,
                                   swa_v_scale=SWA_V_SCALE, device=device)
            swa = DecodeStack(n_max, Hq, Hkv, 1, 1, n_layers=n_swa, full_every=n_swa + 1, ring_capacity=ring,
                              window=window, swa_k_scale=SWA_K_SCALE, swa_v_scale=SWA_V_SCALE, device=device)
            for stack in (full, swa):
                for layer in stack.layers:
                    fill_pool_random(layer.tensors, gen)
            held = torch.cuda.memory_allocated() / 1e9
            q = torch.empty((n_max, 1, Hq, 128), dtype=torch.bfloat16, device=device)
            kn = torch.empty((n_max, 1, Hkv, 128), dtype=torch.bfloat16, device=device)
            vn = torch.empty_like(kn)
            for buf, sid in ((q, synth.S_QUERIES), (kn, synth.S_KEYS), (vn, synth.S_VALUES)):
                synth.normals_device(synth.key(7, sid), 0, buf.numel(), buf.data_ptr(), None, True, stream)
            ctx = torch.full((n_max,), ctx_len, dtype=torch.int32, device=device)
            out = torch.empty((n_max, 1, Hq, 128), dtype=torch.float32, device=device)
            # halvings from the pool's maximum, plus the other format's maximum (equal-batch
            # comparison) and 8 sessions (the 256k step's batch)
            other = int(budget_gb * 1e9 // per_session["fp8" if fmt == "int4" else "int4"])
            sizes = sorted({max(1, n_max >> i) for i in range(12)} | {b for b in (other, 8) if b <= n_max},
                           reverse=True)
            for B in sizes:
                def step(B=B):
                    # model order: every fifth layer is full attention
                    for l in range(n_full + n_swa):
                        st, idx = (full, l // 5) if l % 5 == 4 else (swa, l - (l + 1) // 5)
                        st.decode_layer(idx, q[:B], ctx[:B], out[:B], k_new=kn[:B], v_new=vn[:B])
                for _ in range(warmup):
                    step()
                torch.cuda.synchronize()
                cs = torch.cuda.Stream()
                cs.wait_stream(torch.cuda.current_stream())
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(cs):
                    with torch.cuda.graph(g, stream=cs):
                        step()
                torch.cuda.synchronize()
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(steps)]
                for e0, e1 in evs:
                    e0.record()
                    g.replay()
                    e1.record()
                torch.cuda.synchronize()
                ms = np.array([e0.elapsed_time(e1) for e0, e1 in evs])
                med = float(np.median(ms))
                assert full.read_error() == 0 and swa.read_error() == 0
                result["points"].append({
                    "context": ctx_len, "format": fmt, "sessions_max": n_max, "bytes_per_session": per_session[fmt],
                    "pool_gb_held": round(held, 1), "sessions": B, "ms_per_step": round(med, 3),
                    "session_steps_per_s": round(B / med * 1e3, 1),
                    "p90_over_median": round(float(np.percentile(ms, 90)) / med, 3)})
                del g
            del full, swa, q, kn, vn, out
            torch.cuda.empty_cache()
    pts = result["points"]

    def at(ctx_len, fmt, B=None):
        c = [p for p in pts if p["context"] == ctx_len and p["format"] == fmt]
        return c[0] if B is None else min(c, key=lambda p: abs(p["sessions"] - B))

    summary = {}
    for ctx_len in (65536, 262144):
        i4, f8 = at(ctx_len, "int4"), at(ctx_len, "fp8")
        same_b = at(ctx_len, "int4", f8["sessions"])
        summary[str(ctx_len)] = {
            "sessions_int4": i4["sessions_max"], "sessions_fp8": f8["sessions_max"],
            "sessions_gain": round(i4["sessions_max"] / f8["sessions_max"] - 1, 3),
            "throughput_at_full_memory_gain": round(i4["session_steps_per_s"] / f8["session_steps_per_s"] - 1, 3),
            "fp8_over_int4_step_time_at_equal_batch": round(f8["ms_per_step"] / same_b["ms_per_step"], 3)
            if same_b["sessions"] == f8["sessions"] else None,
            "equal_batch_sessions": f8["sessions"],
            "worst_p90_over_median": max(p["p90_over_median"] for p in pts if p["context"] == ctx_len)}
    result["summary"] = summary
    return result


# ---------------------------------------------------------------- CPU oracle timing

def _oracle_heads_concurrently(calls, threads_total):
    """Run one oracle call per KV head on its own host thread (ctypes releases the GIL), each with
    threads_total // len(calls) oracle threads. Returns (seconds, threads actually busy)."""
    import concurrent.futures

    import oracle

    per = max(1, threads_total // len(calls))
    Os = [oracle.Oracle(threads=per) for _ in calls]
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(len(calls)) as pool:
        list(pool.map(lambda a: a[0](a[1]), zip(calls, Os)))
    return time.perf_counter() - t0, per


class OracleStepSample:
    """The fp64 oracle on a bounded sample of the 256k decode step, on the host's cores: one int4
    layer of one sequence (its 4 KV heads, 5 query rows each, over 262,145 positions of seeded
    random codes) and one window-513 layer of one sequence (4 KV heads, 5 rows each). Each KV head
    is one oracle call on its own host thread; an oracle call threads over its query rows, so
    4 x min(5, cores / 4) threads do the attention (cores() reports that number). A session-step
    is 10 int4 layers and 40 window layers: seconds per session-step = 10 t_int4 + 40 t_window."""

    def __init__(self):
        import synth
        from synth.workloads import config

        w = config(5)
        self.w = w
        self.threads_total = max(1, os.cpu_count() or 1)
        L = int(w.ctx[0]) + 1
        self.L = L
        self.int4 = []
        for h in range(w.Hkv):
            raw = synth.draws(synth.key(99, 10 + h), 0, L * 128 // 4).view(np.uint8)
            kc = np.ascontiguousarray((raw[: L * 128] & 15).reshape(L, 128))
            vc = np.ascontiguousarray((raw[: L * 128] >> 4).reshape(L, 128))
            q = synth.normals(synth.key(99, 20 + h), 0, w.G * 128).reshape(w.G, 128)
            self.int4.append((q, kc, vc))
        self.ks = np.full(L, 0x2E66, np.uint16)
        self.ko = np.full(L, 0xC1A0, np.uint16)
        W = w.window
        self.W = W
        self.swa = []
        for h in range(w.Hkv):
            raw = synth.draws(synth.key(99, 30 + h), 0, W * 128 // 4).view(np.uint8)
            k8 = np.ascontiguousarray((raw[: W * 128] & 0x77).reshape(W, 128))
            v8 = np.ascontiguousarray((raw[: W * 128] >> 1 & 0x77).reshape(W, 128))
            q8 = synth.normals(synth.key(99, 40 + h), 0, w.G * 128).reshape(w.G, 128)
            self.swa.append((q8, k8, v8))

    def cores(self):
        return self.w.Hkv * min(self.w.G, max(1, self.threads_total // self.w.Hkv))

    def layer_seconds(self):
        """(t_int4_layer, t_window_layer) for one sequence, all KV heads."""
        w, L, W = self.w, self.L, self.W
        vis = np.full(w.G, L)
        calls = [lambda O, a=a: O.attention_int4(a[0], vis, a[1], self.ks, self.ko, a[2], self.ks, self.ko,
                                                  128 ** -0.5) for a in self.int4]
        t_int4, _ = _oracle_heads_concurrently(calls, self.threads_total)
        lo = np.zeros(w.G, np.int64)
        hi = np.full(w.G, W - 1, np.int64)
        calls = [lambda O, a=a: O.attention_fp8(a[0], lo, hi, a[1], a[2], 0.01, 0.01, 128 ** -0.5) for a in self.swa]
        t_swa, _ = _oracle_heads_concurrently(calls, self.threads_total)
        return t_int4, t_swa

    def per_session_step(self, t_int4, t_swa):
        return self.w.int4_layers * t_int4 + self.w.swa_layers * t_swa

    def describe(self):
        return (f"fp64 oracle, per sample one int4 layer of one sequence (4 KV heads x 5 query rows over {self.L} "
                f"positions) and one window-513 layer of one sequence (4 KV heads x 5 rows), each KV head an "
                f"oracle call on its own host thread; seconds per session-step = "
                f"{self.w.int4_layers} x int4 layer + {self.w.swa_layers} x window layer")


def oracle_sample(seconds_budget=20.0):
    """cpu_baseline of the kvq arm: OracleStepSample repeated within the budget (at most 4
    samples), the median sample scaled to session-steps/s."""
    smp = OracleStepSample()
    res = []
    t0 = time.perf_counter()
    while True:
        res.append(smp.layer_seconds())
        if time.perf_counter() - t0 > seconds_budget / 2 or len(res) >= 4:
            break
    per = statistics.median([smp.per_session_step(a, b) for a, b in res])
    return {"value": round(1.0 / per, 4), "unit": "session-steps/s", "cores": smp.cores(), "kind": "oracle",
            "sample": smp.describe() + f"; {len(res)} samples, median", "seconds_per_session_step": per}


# ---------------------------------------------------------------- arms

def run_kvq(args, rank, world, local):
    import torch

    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    K, W = args.steps, args.warmup
    total = K + W + 2 * min(K, 64)  # timed, warm-up and end-to-end steps each append one position
    bench = Stack256k(total, device, prologue=args.prologue)
    peak, peak_kind = measured_peak()

    # ---- device-resident timed region: the K steps are captured once into a CUDA graph (as a
    # serving engine would) and replayed. Event-record nodes bracket the int4 layer calls of
    # every 64th step and of the last one: each such node drains the GPU's work queue (several
    # microseconds), so bracketing every call would slow the very steps being timed.
    for t in range(W):
        bench.step(t)
    torch.cuda.synchronize()
    n_int4 = len(bench.int4)

    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None

    sampled = [i for i in range(K) if i % 64 == 63 or i == K - 1]
    evs = [timing_event() for _ in range(2 * n_int4 * len(sampled))]
    if any(e is None for e in evs):
        evs = None
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(K):
                si = sampled.index(i) if (evs is not None and i in sampled) else -1
                bench.step(W + i, None if si < 0 else evs[2 * n_int4 * si: 2 * n_int4 * (si + 1)])
    torch.cuda.synchronize()
    # one untimed replay first: the first launch of a graph also uploads it to the device (the
    # replay rewrites the same cache slots with the same values)
    graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    torch.cuda.nvtx.range_push("timed")
    start.record()
    graph.replay()
    end.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms_local = start.elapsed_time(end)
    err = bench.st.read_error()
    assert err == 0, f"device error word {err:#x}"
    ms, value = aggregate(ms_local, bench.w.B * K, world, device)
    call_bytes = [bench.int4_call_bytes(W + sampled[j // n_int4]) for j in range(n_int4 * len(sampled))]
    if evs is not None:
        call_ms = [evs[2 * j].elapsed_time(evs[2 * j + 1]) for j in range(n_int4 * len(sampled))]
    else:  # no event nodes in graphs on this torch: time the same calls eagerly right after
        call_ms = []
        for j in range(min(n_int4 * K, 100)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            l = sorted(bench.int4)[j % n_int4]
            e0.record()
            bench.st.decode_layer(l, bench.q[W, l], bench.ctx[W], bench.out[l])
            e1.record()
            torch.cuda.synchronize()
            call_ms.append(e0.elapsed_time(e1))
        call_bytes = call_bytes[:len(call_ms)]
    achieved = sum(call_bytes) / (sum(call_ms) * 1e-3) / 1e9
    del graph

    # ---- per-step times: one decode step captured alone, replayed n_dist times with events
    # around each replay (the pages' method times 512 steps per point and reports the slowest
    # tenth against the median)
    n_dist = 512
    g1 = torch.cuda.CUDAGraph()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g1, stream=cap):
            bench.step(W + K - 1)
    torch.cuda.synchronize()
    dist_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dist)]
    for d0, d1 in dist_evs:
        d0.record()
        g1.replay()
        d1.record()
    torch.cuda.synchronize()
    step_ms = np.array([d0.elapsed_time(d1) for d0, d1 in dist_evs])
    step_med = float(np.median(step_ms))
    assert bench.st.read_error() == 0
    del g1

    # ---- end to end: every step copies its inputs from pinned host memory and reads its
    # outputs back, through the same public calls (captured into a graph with the copies)
    Ke = min(K, 64)
    pool = 4
    hq = torch.empty((pool,) + tuple(bench.q.shape[1:]), dtype=torch.bfloat16).pin_memory()
    hk = torch.empty((pool,) + tuple(bench.kn.shape[1:]), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    for i in range(pool):
        hq[i].copy_(bench.q[i])
        hk[i].copy_(bench.kn[i])
        hv[i].copy_(bench.vn[i])
    hout = torch.empty((Ke,) + tuple(bench.out.shape), dtype=torch.float32).pin_memory()
    h2d = hq[0].numel() * 2 + hk[0].numel() * 2 + hv[0].numel() * 2
    d2h = hout[0].numel() * 4
    base = W + K
    g2 = torch.cuda.CUDAGraph()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g2, stream=cap):
            for i in range(Ke):
                t_ = base + i
                bench.q[t_].copy_(hq[i % pool], non_blocking=True)
                bench.kn[t_].copy_(hk[i % pool], non_blocking=True)
                bench.vn[t_].copy_(hv[i % pool], non_blocking=True)
                bench.step(t_)
                hout[i].copy_(bench.out, non_blocking=True)
    torch.cuda.synchronize()
    g2.replay()  # untimed: the graph's upload to the device (same copies and slots as the timed replay)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g2.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    _, e2e_value = aggregate(e0.elapsed_time(e1), bench.w.B * Ke, world, device)
    assert bench.st.read_error() == 0
    del g2
    launches_per_step = bench.launches_per_step()
    del bench
    torch.cuda.empty_cache()

    sec = run_64k(device) if rank == 0 else None
    verify = run_verify(device) if rank == 0 else None
    cfg2 = run_config2(device) if rank == 0 else None
    cpu = oracle_sample() if rank == 0 else None

    if rank == 0:
        frac = achieved / peak
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "session-steps/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u4", "data": "synthetic",
            "config": step_config(args, world),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(frac, 4), "traffic": attn_traffic(int(np.mean(call_bytes))),
                         "traffic_how": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the attention kernel "
                                        "on the 64k workload, scaled to this call by algorithmic bytes "
                                        "(one capture, cold cache); null once its sources changed",
                         "peak_kind": peak_kind,
                         "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
                         "kernel": "kvq_decode_attn_int4 call (query prologue/append + split-K attention + combine kernels)",
                         "bytes_per_call": int(np.mean(call_bytes)), "avg_call_us": round(1e3 * np.mean(call_ms), 2)},
            "at_64k": sec,
            "step_ms_median": round(step_med, 4),
            "p90_over_median": round(float(np.percentile(step_ms, 90)) / step_med, 4),
            "step_distribution": f"{n_dist} replays of one decode step captured alone, CUDA events around each",
            "verify": verify,
            "config2": cfg2,
            "e2e": {"value": round(e2e_value, 2), "unit": "session-steps/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": Ke,
                    "how": "per step: q, k_new, v_new of all 50 layers copied from pinned host memory, the step, "
                           "all outputs copied back to pinned host memory; captured in one CUDA graph, "
                           "replayed once untimed (its upload to the device), then timed"},
            "timing": "K steps captured in one CUDA graph, replayed once untimed (its upload to the device), "
                      "then replayed timed; CUDA events on the replay stream; "
                      "int4 call durations from event-record nodes inside the graph around the int4 calls of "
                      "every 64th timed step and the last one",
            "int4_calls_timed": len(call_ms),
            "cpu_baseline": {k: v for k, v in cpu.items() if k != "seconds_per_session_step"},
            "gpu_launches": launches_per_step * K,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)


def step_config(args, world):
    """The `config` of both arms' JSON line: the 256k decode step."""
    return {"workload": "decode step at 256k: 8 sequences x 262,144 context, 50 layers "
                        "(10 rotated int4 + 40 FP8 window 513), 20/4 heads x 128, bf16 inputs, 1 query row",
            "prologue": args.prologue,
            "global_batch": 8 * world, "seq_len": int(bench_ctx0()), "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (11.4 GB of int4 cache read per step)"}


def bench_ctx0():
    from synth.workloads import config
    return config(5).ctx[0]


def run_reference(args, rank, world):
    """The oracle as it stands, on the machine's host cores: each step is one OracleStepSample (one
    int4 layer and one window layer of one sequence, all KV heads), the same scope as the kvq
    arm's cpu_baseline; the value is session-steps/s; rank 0 only."""
    if rank != 0:
        return
    smp = OracleStepSample()
    for _ in range(args.warmup):
        smp.layer_seconds()
    per = []
    for _ in range(args.steps):
        per.append(smp.per_session_step(*smp.layer_seconds()))
    per_step = float(np.mean(per))
    value = 1.0 / per_step
    sample = smp.describe() + "; one sample per step"
    line = {"metric": METRIC, "value": round(value, 5), "unit": "session-steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": step_config(args, world),
            "cpu_baseline": {"value": round(value, 5), "unit": "session-steps/s", "cores": smp.cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "session-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--prologue", default="matrix", choices=["matrix", "fwht"],
                    help="Q/K prologue of the int4 layers: the folded 128x128 matrices (default) or the "
                         "fast Walsh-Hadamard form (second codec specification)")
    ap.add_argument("--sequences", type=int, default=None,
                    help="--only swa: this many sequences instead of the 256k step's 8")
    ap.add_argument("--layers", type=int, default=None, help="--only swa: this many window layers instead of 40")
    ap.add_argument("--only", default=None, choices=["64k", "swa", "ab", "capacity", "verify", "config2"],
                    help="run only the 64k single-layer int4 point, only the 40 window layers of the 256k "
                         "step (small cases for profiling), the A/B of full-layer formats (ab), the "
                         "capacity and throughput sweep of a fixed KV pool (capacity), the speculative "
                         "verify workload at S = 1..8 (verify), or the 16 x 8,192 layer with L2 flushed "
                         "between calls (config2)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.only == "64k":
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_64k(f"cuda:{local}", steps=args.steps, warmup=args.warmup)), flush=True)
    elif args.only == "capacity":
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_capacity(f"cuda:{local}", steps=args.steps, warmup=args.warmup)), flush=True)
    elif args.only == "ab":
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_ab(f"cuda:{local}", steps=args.steps, warmup=args.warmup)), flush=True)
    elif args.only == "verify":
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_verify(f"cuda:{local}", steps=args.steps, warmup=args.warmup,
                                    S_values=tuple(range(1, 9)))), flush=True)
    elif args.only == "config2":
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_config2(f"cuda:{local}", steps=args.steps, warmup=args.warmup)), flush=True)
    elif args.only == "swa":
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_swa(f"cuda:{local}", steps=args.steps, warmup=args.warmup, sequences=args.sequences,
                                 layers=args.layers)), flush=True)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_kvq(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
