#!/usr/bin/env python
"""Benchmark of the OSCAR INT2 KV-cache serving path (write path + fused paged
decode attention) on synthetic Qwen3-shaped attention layers.

A step is one decode step of one layer for the whole batch through
oscar_decode_step: one new token per request appended (ring write; the token
leaving the recent window rotated, clipped, quantised and packed) and one
decode query over the cache that then holds it (query rotation, split-K INT2 +
BF16 attention, merge and un-rotation), the append done by CTAs of the decode
launch. The same step as two calls (quant_append, then decode_attn) is timed
beside it. Inputs are resident in device memory before timing starts.

Default workload: Qwen3-8B layer shape (32 query / 8 KV heads, d = 128), batch
1 at 32768 tokens. Its cache (25.6 MB) fits in L2, so the timed loop cycles
through enough independent layer caches to exceed 4x the L2 size, as a model
with that many layers would. The Qwen3-32B-shaped batch-28 x 100000-token
layer (2.15 GB) is measured as well and reported under "extra".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl oscar|reference]

Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); timings are the max over ranks.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import WORKLOADS, draw_kv, draw_page_pool, draw_queries, draw_ragged_lengths  # noqa: E402

METRIC = "paged INT2 decode-attn µs/step & HBM GB/s (% of peak), bs1@32k and bs28@100k"
D = 128
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

# GB300's nominal HBM3e bandwidth, reported beside the measured denominator
NOMINAL_HBM_GBS = 7900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings, returned on every rank (the
    replicas run concurrently, so the job takes as long as its slowest rank)."""
    if not dist:
        return [float(v) for v in values]
    dev = device if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


KERNEL_SOURCES = {"decode": ("decode_attn.cu", "oscar_internal.cuh", "token_quant.cuh"),
                  "prefill": ("prefill_append.cu", "oscar_internal.cuh")}


def source_hash(kind="decode"):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "bit_rotated_kv_oscar_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kind="decode"):
    """DRAM bytes per launch of the kernel from a committed ncu summary, if it was
    taken on the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "%s_traffic.json" % kind)
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("source_hash") != source_hash(kind):
            return None
        return t.get("bytes_per_launch", {}).get(workload)
    except Exception:
        return None


# ---------------------------------------------------------------------------
# one workload: layers, caches, inputs
# ---------------------------------------------------------------------------

class Workload:
    def __init__(self, name, device, n_steps_total, rank=0, min_layers=None, batch_override=0):
        from bit_rotated_kv_oscar_gb300 import abi
        from bit_rotated_kv_oscar_gb300.cache import PagedCache
        from bit_rotated_kv_oscar_gb300.calibrate import calibrate

        spec = WORKLOADS[name]
        if batch_override:
            spec = dataclasses.replace(spec, batch=batch_override)
        self.spec, self.name, self.device = spec, name, device
        hq, hkv, S, W, B = spec.num_q_heads, spec.num_kv_heads, spec.sink, spec.recent, spec.batch
        self.B = B
        seed = spec.seed + 1000 * rank
        self.lengths = draw_ragged_lengths(seed, B, spec.context_min, spec.context)
        max_len = int(self.lengths.max()) + n_steps_total + 16
        max_pages = (max_len + 15) // 16
        # offline calibration on 2048 synthetic calibration tokens
        q_cal = draw_queries(seed, 900, spec.calib_tokens, hq, hkv, D).numpy()
        k_cal, v_cal = (t.numpy() for t in draw_kv(seed, 900, spec.calib_tokens, hkv, D, spec.token_spikes))
        cal = calibrate(q_cal, k_cal, v_cal, clip_percentile_k=spec.clip_percentile_k,
                        clip_percentile_v=spec.clip_percentile_v)
        self.cfg = abi.make_config(hq, hkv, S, W, B, max_pages, group_size=spec.group_size)
        num_pages = B * max_pages
        # cache bytes of one layer at the starting lengths
        int2_tok = np.maximum(self.lengths - W, S) - S
        per_layer = int(hkv * spec.int2_token_bytes * int2_tok.sum())
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n_layers = 1 if per_layer > 4 * l2 else int(math.ceil(4 * l2 / max(per_layer, 1)))
        if min_layers:
            n_layers = max(n_layers, min_layers)
        self.layers = []
        for li in range(n_layers):
            ctx = abi.Context(self.cfg)
            ctx.load_rotations(cal["R_K"], cal["R_V"], cal["clip_K"], cal["clip_V"])
            cache = PagedCache(ctx, num_pages, device=device,
                               page_order=draw_page_pool(seed + li, num_pages, spec.shuffled_pages))
            for b in range(B):
                cache.reserve(b, max_len, upload=False)
            cache.upload()
            self.layers.append((ctx, cache))
        self._populate()
        # per-step inputs (a small ring of distinct draws, resident on the device)
        self.n_inputs = 8
        self.q = [draw_queries(seed, 100 + i, B, hq, hkv, D, device=device).to(torch.bfloat16).contiguous()
                  for i in range(self.n_inputs)]
        kv = [draw_kv(seed, 100 + i, B, hkv, D, spec.token_spikes, device=device) for i in range(self.n_inputs)]
        self.k = [a.to(torch.bfloat16).view(B, 1, hkv, D).contiguous() for a, _ in kv]
        self.v = [b_.to(torch.bfloat16).view(B, 1, hkv, D).contiguous() for _, b_ in kv]
        self.o = torch.empty(B, hq, D, device=device)
        self.per_layer_bytes = per_layer

    def _populate(self):
        """Fill every request of every layer: the longest request of layer 0 goes
        through quant_append (the product's write path) in chunks; its pages,
        window rows and state are then copied to the other requests and layers
        (distinct addresses, same contents)."""
        spec, B = self.spec, self.B
        ctx0, c0 = self.layers[0]
        hkv = spec.num_kv_heads
        b0 = int(np.argmax(self.lengths))
        L0 = int(self.lengths[b0])
        chunk = 16384
        pos = 0
        while pos < L0:
            n = min(chunk, L0 - pos)
            k, v = draw_kv(spec.seed, 10_000 + pos // chunk, n, hkv, D, spec.token_spikes, device=self.device)
            ctx0.quant_append(c0.page_table[b0:], c0.state[b0:], k.to(torch.bfloat16).contiguous(),
                              v.to(torch.bfloat16).contiguous(), 1, n)
            pos += n
        torch.cuda.synchronize()
        from bit_rotated_kv_oscar_gb300 import abi

        bb = abi.page_block_bytes(spec.group_size)
        pool0 = c0.pool.view(-1, hkv, bb)
        win0 = c0.window.view(B, hkv, 2, spec.sink + spec.recent, D)
        st0 = c0.state[b0].clone()
        S, W = spec.sink, spec.recent
        src_pages = torch.as_tensor(c0.page_table_host[b0].astype(np.int64), device=self.device)
        for li, (ctx, cache) in enumerate(self.layers):
            pool = cache.pool.view(-1, hkv, bb)
            win = cache.window.view(B, hkv, 2, S + W, D)
            for b in range(B):
                if li == 0 and b == b0:
                    continue
                L = int(self.lengths[b])
                npg = (L + 15) // 16
                dst = torch.as_tensor(cache.page_table_host[b, :npg].astype(np.int64), device=self.device)
                pool[dst] = pool0[src_pages[:npg]]
                win[b].copy_(win0[b0])
                E = max(S, L - W)
                cache.state[b] = torch.tensor([L, E, b, 0], dtype=torch.int32, device=self.device)
        torch.cuda.synchronize()

    def decode_bytes(self, extra_tokens):
        """Algorithmic HBM bytes of one decode_attn call with every request extra_tokens longer."""
        s = self.spec
        L = self.lengths + extra_tokens
        E = np.maximum(L - s.recent, s.sink)
        n_int2 = E - s.sink
        n_bf16 = np.minimum(L, s.sink) + (L - E)
        pages = (E + 15) // 16
        b = s.num_kv_heads * (s.int2_token_bytes * n_int2 + 512 * n_bf16) + 4 * pages
        return float(b.sum() + self.B * s.num_q_heads * D * (2 + 4))

    def append_bytes(self):
        """Algorithmic HBM bytes of one single-token quant_append for the batch:
        read the new K/V (512 B per head), read the evicted ring token (512 B),
        write its INT2 codes + metadata (96 B for groups of 32) and the new ring
        row (512 B)."""
        s = self.spec
        return float(self.B * s.num_kv_heads * (512 + 512 + s.int2_token_bytes + 512))

    def decode_only(self, i, stream):
        ctx, cache = self.layers[i % len(self.layers)]
        j = i % self.n_inputs
        ctx.decode_attn(self.q[j], cache.page_table, cache.state, self.o, self.B, stream)

    def decode_timed(self, i, stream, ev_before, ev_after):
        """decode_attn with the split-K attention kernel bracketed by two events."""
        ctx, cache = self.layers[i % len(self.layers)]
        j = i % self.n_inputs
        ctx.decode_attn_timed(self.q[j], cache.page_table, cache.state, self.o, self.B, ev_before, ev_after,
                              stream)

    def step(self, i, stream):
        """One decode step: oscar_decode_step (the append inside the decode launches)."""
        ctx, cache = self.layers[i % len(self.layers)]
        j = i % self.n_inputs
        ctx.decode_step(cache.page_table, cache.state, self.q[j], self.k[j], self.v[j], self.o, self.B, stream)

    def step_two_calls(self, i, stream):
        """The same step as quant_append followed by decode_attn."""
        ctx, cache = self.layers[i % len(self.layers)]
        j = i % self.n_inputs
        ctx.quant_append(cache.page_table, cache.state, self.k[j], self.v[j], self.B, 1, stream)
        ctx.decode_attn(self.q[j], cache.page_table, cache.state, self.o, self.B, stream)


def run_oscar(name, args, device, rank, world, dist, clocks_index, with_e2e=True):
    n_total = 2 * args.warmup + 6 * args.steps + 4096 + 64
    wl = Workload(name, device, n_total, rank, batch_override=getattr(args, 'batch', 0))
    stream = torch.cuda.current_stream(device)
    # warm-up: at least W steps and about half a second under load
    i = 0
    t0 = time.time()
    sampler = ClockSampler(clocks_index)
    sampler.start()
    while i < args.warmup or time.time() - t0 < 0.5:
        wl.step(i, stream)
        i += 1
        if i % 256 == 0:
            torch.cuda.synchronize()
        if i > n_total - 5 * args.steps - 2 * args.warmup - 32:
            break
    torch.cuda.synchronize()
    # three CUDA graphs, captured once and warmed once:
    #   g_time - K decode steps (oscar_decode_step): the timed region, the headline value;
    #   g_two  - the same K steps as quant_append + decode_attn, timed after it;
    #   g_dec  - K decode_attn calls over the same layers (decode leaves the cache
    #            unchanged), timed last: the decode call's duration
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    graphs = []
    for fn in (wl.step, wl.step_two_calls, wl.decode_only):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for k in range(args.steps):
                    fn(i + k, cap)
        graphs.append(g)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    i += 2 * args.steps
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    # NVTX ranges name the replays for profilers (ncu --nvtx --nvtx-include
    # "timed_steps/"); they are host-side markers outside the events
    for n, g in enumerate(graphs):
        torch.cuda.nvtx.range_push(("timed_steps", "two_call_steps", "decode_calls")[n])
        ev[2 * n].record(stream)
        g.replay()
        ev[2 * n + 1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = ev[0].elapsed_time(ev[1])
    two_ms = ev[2].elapsed_time(ev[3]) / args.steps
    dec_ms = ev[4].elapsed_time(ev[5]) / args.steps
    # the append kernel's share of a two-call step
    app_ms = max(two_ms - dec_ms, 0.0)
    warm_done = i
    i += 2 * args.steps
    # the split-K attention kernel alone: eager decode calls, each bracketing that
    # launch with its own event pair (layers cycled as in the timed graphs)
    n_k = min(args.steps, 64)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_k)]
    torch.cuda.nvtx.range_push("decode_timed")
    for k in range(n_k):
        wl.decode_timed(i + k, stream, *kev[k])
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    kern_ms = sum(a.elapsed_time(b) for a, b in kev) / n_k
    total_ms, app_ms, dec_ms, kern_ms, two_ms = max_over_ranks([total_ms, app_ms, dec_ms, kern_ms, two_ms], dist,
                                                               device)
    us_step = total_ms * 1000.0 / args.steps
    mid = warm_done + args.steps // 2
    dbytes = wl.decode_bytes(mid // len(wl.layers))
    res = {
        "workload": name, "us_per_step": us_step, "decode_us": dec_ms * 1000.0, "kernel_us": kern_ms * 1000.0,
        "kernel_bytes": dbytes - wl.B * wl.spec.num_q_heads * D * 6,
        "append_us": app_ms * 1000.0, "two_call_us_per_step": two_ms * 1000.0,
        "decode_bytes": dbytes, "append_bytes": wl.append_bytes(),
        "layers_cycled": len(wl.layers), "per_layer_bytes": wl.per_layer_bytes, "clocks": clocks,
        "batch": wl.B, "lengths": [int(x) for x in wl.lengths[:4]],
    }
    if with_e2e:
        res["e2e"] = run_e2e(wl, args, device, i, dist)
    return res


def run_e2e(wl, args, device, i0, dist):
    """Same steps through the public API with host buffers: per step one
    oscar_decode_step_host call copies the new q / k / v host->device from pinned
    memory, appends, decodes and copies o back."""
    stream = torch.cuda.current_stream(device)
    # each step's q, k, v packed in one pinned host buffer: one host->device copy
    nq, nk, nv = wl.q[0].numel(), wl.k[0].numel(), wl.v[0].numel()
    hbuf = [torch.cat([wl.q[j].reshape(-1), wl.k[j].reshape(-1), wl.v[j].reshape(-1)]).cpu().pin_memory()
            for j in range(wl.n_inputs)]
    dbuf = torch.empty(nq + nk + nv, dtype=wl.q[0].dtype, device=device)
    ho = torch.empty(wl.o.shape, dtype=wl.o.dtype).pin_memory()
    h2d = dbuf.numel() * dbuf.element_size()
    d2h = ho.numel() * 4

    def one(k):
        ctx, cache = wl.layers[k % len(wl.layers)]
        j = k % wl.n_inputs
        ctx.decode_step_host(cache.page_table, cache.state, hbuf[j], dbuf, wl.o, ho, wl.B, stream)

    for k in range(max(3, args.warmup)):
        one(i0 + k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    base = i0 + max(3, args.warmup)
    start.record(stream)
    for k in range(args.steps):
        one(base + k)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    ms = max_over_ranks([ms], dist, device)[0]
    return {"value": ms * 1000.0 / args.steps, "unit": "us/step", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h}


def run_prefill(args, device, rank, dist):
    """131072-token prefill quant-append into a fresh request, then 16 requests
    sharing its first 65536 tokens through aliased pages, each with a private
    4096-token suffix, decoded for one step."""
    from bit_rotated_kv_oscar_gb300 import abi
    from bit_rotated_kv_oscar_gb300.cache import PagedCache
    from bit_rotated_kv_oscar_gb300.calibrate import calibrate

    spec = WORKLOADS["prefill_128k_prefix16"]
    hq, hkv, S, W = spec.num_q_heads, spec.num_kv_heads, spec.sink, spec.recent
    n, fork, suf, nreq = spec.context, spec.prefix_shared, spec.suffix, spec.batch
    seed = spec.seed + 1000 * rank
    q_cal = draw_queries(seed, 900, spec.calib_tokens, hq, hkv, D).numpy()
    k_cal, v_cal = (t.numpy() for t in draw_kv(seed, 900, spec.calib_tokens, hkv, D))
    cal = calibrate(q_cal, k_cal, v_cal)
    max_pages = (n + 15) // 16 + 8
    cfg = abi.make_config(hq, hkv, S, W, nreq + 1, max_pages)
    ctx = abi.Context(cfg)
    ctx.load_rotations(cal["R_K"], cal["R_V"], cal["clip_K"], cal["clip_V"])
    num_pages = (n + 15) // 16 + nreq * (suf // 16 + 2) + 16
    cache = PagedCache(ctx, num_pages, device=device,
                       page_order=draw_page_pool(seed, num_pages, True))
    cache.reserve(0, n)
    k, v = (t.to(torch.bfloat16).view(1, n, hkv, D).contiguous()
            for t in draw_kv(seed, 1, n, hkv, D, device=device))
    stream = torch.cuda.current_stream(device)
    fresh = torch.tensor([0, S, 0, 0], dtype=torch.int32, device=device)
    times, ktimes = [], []
    for it in range(max(3, args.warmup) + 2 * args.steps):
        cache.state[0].copy_(fresh)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # keep the device busy while the host encodes and launches, so the events
        # bracket device time only
        torch.cuda._sleep(200000)
        if it < max(3, args.warmup) + args.steps:
            # the whole call (tensor-core kernel + per-token tail kernel)
            e0.record(stream)
            ctx.quant_append(cache.page_table, cache.state, k, v, 1, n, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= max(3, args.warmup):
                times.append(e0.elapsed_time(e1))
        else:
            # the tensor-core kernel alone
            ctx.quant_append_timed(cache.page_table, cache.state, k, v, 1, n, e0, e1, stream)
            torch.cuda.synchronize()
            ktimes.append(e0.elapsed_time(e1))
    pre_us = float(np.mean(times)) * 1000.0
    pre_kernel_us = float(np.mean(ktimes)) * 1000.0
    n_int2 = max(n - W, S) - S
    tb = spec.int2_token_bytes
    pre_bytes = float(n * hkv * 2 * D * 2 + n_int2 * hkv * tb + (S + W) * hkv * 2 * D * 2)
    # 16 forks at 65536 tokens with private suffixes
    for r in range(1, nreq + 1):
        cache.fork(0, r, fork)
        cache.reserve(r, fork + suf, upload=False)
    cache.upload()
    ks, vs = (t.to(torch.bfloat16).view(nreq, suf, hkv, D).contiguous()
              for t in draw_kv(seed, 2, nreq * suf, hkv, D, device=device))
    ctx.quant_append(cache.page_table[1:], cache.state[1:], ks, vs, nreq, suf, stream)
    q = draw_queries(seed, 3, nreq, hq, hkv, D, device=device).to(torch.bfloat16).contiguous()
    o = torch.empty(nreq, hq, D, device=device)
    def graph_us(call):
        """Mean duration of one call, timed over a CUDA graph of args.steps calls."""
        for _ in range(max(3, args.warmup)):
            call(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for _ in range(args.steps):
                    call(cap)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / args.steps

    # every fork reads the shared pages itself, then the shared range once per pack
    dec_us = graph_us(lambda st: ctx.decode_attn(q, cache.page_table[1:], cache.state[1:], o, nreq, st))
    shared_us = graph_us(lambda st: ctx.decode_attn_shared_prefix(q, cache.page_table[1:], cache.state[1:], fork,
                                                                  o, nreq, st))
    L = fork + suf
    E = L - W
    logical = float(nreq * (hkv * (tb * (E - S) + 512 * (S + W)) + 4 * ((E + 15) // 16)) + nreq * hq * D * 6)
    unique = float(hkv * tb * (fork - S) + nreq * hkv * (tb * (E - fork) + 512 * (S + W)) + nreq * hq * D * 6)
    pre_us, pre_kernel_us, dec_us, shared_us = max_over_ranks([pre_us, pre_kernel_us, dec_us, shared_us], dist,
                                                              device)
    # the tensor-core kernel's share of the bytes: the K / V of the tokens going
    # straight to INT2 and their codes + metadata
    pre_kernel_bytes = float(n_int2 * hkv * (2 * D * 2 + tb))
    return {"prefill_tokens": n, "prefill_us": pre_us, "prefill_bytes": pre_bytes,
            "prefill_kernel_us": pre_kernel_us, "prefill_kernel_bytes": pre_kernel_bytes,
            "prefix_decode_us": dec_us, "prefix_shared_decode_us": shared_us,
            "prefix_logical_bytes": logical, "prefix_unique_bytes": unique}


def footprint(name):
    """Cache bytes of one layer of a workload: BF16 cache against this INT2 cache."""
    s = WORKLOADS[name]
    L = s.context
    bf16 = s.batch * L * s.num_kv_heads * 2 * D * 2
    n_int2 = max(L - s.recent, s.sink) - s.sink
    pages = (L + 15) // 16
    block = 1024 + 128 * (D // s.group_size)   # one (page, KV head) block, include/oscar.h
    oscar = s.batch * (pages * s.num_kv_heads * block + (s.sink + s.recent) * s.num_kv_heads * 2 * D * 2)
    bits = {}
    for g in (32, 64, 128):
        bits["G%d_bits_per_int2_element" % g] = 2 + 32 / g
    # stored bits per cached element (K and V, INT2 pages and the BF16 window)
    stored = 8.0 * oscar / (s.batch * L * s.num_kv_heads * 2 * D)
    return {"workload": name, "group": s.group_size, "sink": s.sink, "recent": s.recent,
            "bf16_bytes": bf16, "oscar_bytes": oscar, "ratio": round(bf16 / oscar, 3),
            "stored_bits_per_element": round(stored, 3), "int2_tokens_per_request": n_int2, **bits}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

def oracle_step_sample(name, kv_heads_in_sample=1, seed_offset=0, runs=1):
    """Time one oracle decode step (append of one token + float64 attention over
    the whole cache) for request 0 restricted to `kv_heads_in_sample` KV heads,
    `runs` times on the same cache. Returns (seconds per run, scale) where scale
    converts one run to one full batch step."""
    import oracle
    from oracle import OracleCache, decode_attention, next_state

    spec = WORKLOADS[name]
    seed = spec.seed + seed_offset
    hkv = kv_heads_in_sample
    g = spec.gqa
    L = int(draw_ragged_lengths(seed, spec.batch, spec.context_min, spec.context)[0])
    q_cal = draw_queries(seed, 900, 512, g * hkv, hkv, D).numpy()
    k_cal, v_cal = (t.numpy() for t in draw_kv(seed, 900, 512, hkv, D))
    cal = oracle.calibrate(q_cal, k_cal, v_cal)
    k, v = (t.numpy() for t in draw_kv(seed, 1, L + 1, hkv, D))
    q = draw_queries(seed, 2, 1, g * hkv, hkv, D).numpy()[0]
    L0, E0 = next_state(0, spec.sink, L, spec.recent, spec.sink)
    cache = OracleCache(cal["R_K32"], cal["R_V32"], cal["clip_K32"], cal["clip_V32"], spec.sink)
    cache.build(k, v, L0, E0)
    times = []
    for _ in range(runs):
        t0 = time.perf_counter()
        # the appended token evicts one ring entry: rotate + quantise it (K and V), then attend
        p = max(E0, spec.sink)
        for x, r, c in ((k, cal["R_K32"], cal["clip_K32"]), (v, cal["R_V32"], cal["clip_V32"])):
            xr = np.einsum("nhi,hij->nhj", x[p:p + 1].astype(np.float64), r.astype(np.float64))
            oracle.quantize_groups(xr.astype(np.float32), c.reshape(1, -1, 1))
        decode_attention(q, cache)
        times.append(time.perf_counter() - t0)
    scale = spec.batch * spec.num_kv_heads / hkv
    return (times[0] if runs == 1 else times), scale


def oracle_prefill_sample(tokens=8192, runs=3):
    """Time the oracle's write path of the 131072-token prefill (rotate in float64,
    clip, quantise, pack into page blocks; K and V) on `tokens` tokens of one KV
    head, `runs` times. Returns (seconds per run, scale to the whole prefill)."""
    import oracle

    spec = WORKLOADS["prefill_128k_prefix16"]
    q_cal = draw_queries(spec.seed, 900, 512, spec.gqa, 1, D).numpy()
    k_cal, v_cal = (t.numpy() for t in draw_kv(spec.seed, 900, 512, 1, D))
    cal = oracle.calibrate(q_cal, k_cal, v_cal)
    k, v = (t.numpy() for t in draw_kv(spec.seed, 1, tokens, 1, D))
    times = []
    for _ in range(runs):
        t0 = time.perf_counter()
        out = []
        for x, r, c in ((k, cal["R_K32"], cal["clip_K32"]), (v, cal["R_V32"], cal["clip_V32"])):
            xr = np.einsum("nhi,hij->nhj", x.astype(np.float64), r.astype(np.float64))
            out.append(oracle.quantize_groups(xr.astype(np.float32), c.reshape(1, -1, 1)))
        (kc, ks, kz), (vc, vs, vz) = out
        npg = tokens // 16
        oracle.encode_page_block(kc[:, 0].reshape(npg, 16, D), vc[:, 0].reshape(npg, 16, D),
                                 ks[:, 0].reshape(npg, 16, -1), kz[:, 0].reshape(npg, 16, -1),
                                 vs[:, 0].reshape(npg, 16, -1), vz[:, 0].reshape(npg, 16, -1))
        times.append(time.perf_counter() - t0)
    return times, spec.context / tokens * spec.num_kv_heads


def blas_threads():
    """Threads of the BLAS numpy is linked against (threadpoolctl when present,
    else the OpenBLAS entry point found among the loaded libraries), or None."""
    try:
        import threadpoolctl
        info = [d for d in threadpoolctl.threadpool_info() if d.get("user_api") == "blas"]
        if info:
            return int(info[0]["num_threads"])
    except Exception:
        pass
    try:
        import ctypes
        libs = set()
        with open("/proc/self/maps") as f:
            for line in f:
                path = line.split()[-1]
                if "openblas" in path.lower() and ".so" in path:
                    libs.add(path)
        for path in libs:
            lib = ctypes.CDLL(path)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                        "openblas_get_num_threads"):
                fn = getattr(lib, sym, None)
                if fn is not None:
                    return int(fn())
    except Exception:
        pass
    return None


def workload_config(name, world):
    """The JSON line's config of a workload (both arms)."""
    spec = WORKLOADS[name]
    return {"workload": name, "batch": spec.batch, "context": spec.context,
            "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads, "head_dim": D,
            "page": spec.page_size, "group": spec.group_size, "sink": spec.sink,
            "recent": spec.recent, "parallelism": "replicas x%d" % world}


def run_reference(args, name, rank, world=1):
    """The oracle as the reference arm: each step one bounded sample."""
    cores = os.cpu_count()
    times = []
    for k in range(args.warmup + args.steps):
        dt, scale = oracle_step_sample(name, 1, seed_offset=k)
        if k >= args.warmup:
            times.append(dt * scale)
    us = float(np.mean(times)) * 1e6
    sample = "per step: 1 of %d KV heads of request 0 (oracle decode step: append + float64 attention " \
             "over the whole cache), scaled to the full batch" % WORKLOADS[name].num_kv_heads
    return {
        "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference", "config": dict(workload_config(name, world), host="oracle on the host cores"),
        "cpu_baseline": {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="oscar", choices=["oscar", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_bs1_32k")
    ap.add_argument("--extra", default="qwen3_32b_bs28_100k,qwen3_8b_bs16_ragged,qwen3_32b_bs28_100k_pages",
                    help="further decode workloads, comma separated ('' to skip)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill / prefix-sharing measurement")
    ap.add_argument("--prefill-only", action="store_true",
                    help="measure only the prefill / prefix-sharing workload (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, args.workload, rank, world)))
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from bit_rotated_kv_oscar_gb300 import build as _b
    if rank == 0 or not os.path.exists(_b.LIB):
        _b.build()
    if dist:
        dist.barrier()
    peak, peak_kind = peaks()
    if args.prefill_only:
        pre = run_prefill(args, device, rank, dist)
        if rank == 0:
            print(json.dumps({"prefill_only": True, **pre}))
        if dist:
            dist.destroy_process_group()
        return
    main_res = run_oscar(args.workload, args, device, rank, world, dist, local)
    extras = []
    if args.extra:
        for name in args.extra.split(","):
            r = run_oscar(name, args, device, rank, world, dist, local, with_e2e=False)
            extras.append(r)
    pre = None if args.no_prefill else run_prefill(args, device, rank, dist)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        ts, scale = oracle_step_sample(args.workload, 2, runs=3)
        pts, pscale = oracle_prefill_sample()
        cpu = {"value": float(np.median(ts)) * scale * 1e6, "unit": "us/step", "cores": os.cpu_count(),
               "blas_threads": blas_threads(), "kind": "oracle", "runs": 3, "statistic": "median",
               "sample": "one decode step (append + float64 attention over the whole cache) of KV heads "
                         "0-1 of request 0, scaled to all %d KV heads x %d requests; median of 3" %
                         (WORKLOADS[args.workload].num_kv_heads, WORKLOADS[args.workload].batch),
               "prefill_us": round(float(np.median(pts)) * pscale * 1e6, 1),
               "prefill_sample": "131072-token prefill write path (float64 rotation, clip, quantise, pack; "
                                 "K and V): 8192 tokens of 1 of 8 KV heads, scaled by %d; median of 3" % pscale}

    def roof(r):
        # the dominant kernel: split-K attention over the paged cache; algorithmic
        # bytes = INT2 codes + metadata (96 B per token and KV head for groups of 32,
        # 80 B for groups of 64), the BF16 window
        # (512 B per token and KV head) and the page table (4 B per page)
        achieved = r["kernel_bytes"] / (r["kernel_us"] * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(r["workload"]),
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "kernel": "oscar_decode_kernel", "launch_us": round(r["kernel_us"], 3),
                "algorithmic_bytes_per_launch": r["kernel_bytes"]}

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(main_res["us_per_step"], 3), "unit": "us/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(main_res["us_per_step"] / 1000.0, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 hi+lo q~ x u2 codes (mma.sync), f32 accumulate", "data": "synthetic",
            "config": dict(workload_config(args.workload, world),
                           l2="inputs larger than L2: %d independent layer caches cycled" % main_res["layers_cycled"]),
            "decode_us": round(main_res["decode_us"], 3), "append_us": round(main_res["append_us"], 3),
            "two_call_us_per_step": round(main_res["two_call_us_per_step"], 3),
            "decode_gbs": round(main_res["decode_bytes"] / (main_res["decode_us"] * 1e-6) / 1e9, 1),
            "append_gbs": round(main_res["append_bytes"] / (max(main_res["append_us"], 1e-3) * 1e-6) / 1e9, 1),
            "roofline": roof(main_res),
            "cpu_baseline": cpu,
            "e2e": main_res["e2e"],
            "gpu_launches": 3 * args.steps,
            "clocks": main_res["clocks"],
            "extra": [],
        }
        for r in extras:
            es = WORKLOADS[r["workload"]]
            out["extra"].append({
                "workload": r["workload"], "group": es.group_size, "sink": es.sink, "recent": es.recent,
                "us_per_step": round(r["us_per_step"], 3), "two_call_us_per_step": round(r["two_call_us_per_step"], 3),
                "decode_us": round(r["decode_us"], 3), "append_us": round(r["append_us"], 3),
                "decode_gbs": round(r["decode_bytes"] / (r["decode_us"] * 1e-6) / 1e9, 1),
                "append_gbs": round(r["append_bytes"] / (max(r["append_us"], 1e-3) * 1e-6) / 1e9, 1),
                "roofline": roof(r), "clocks": r["clocks"], "layers_cycled": r["layers_cycled"],
            })
        if pre is not None:
            ach = pre["prefill_bytes"] / (pre["prefill_us"] * 1e-6) / 1e9
            kach = pre["prefill_kernel_bytes"] / (pre["prefill_kernel_us"] * 1e-6) / 1e9
            out["prefill"] = {
                "workload": "prefill_128k_prefix16", "tokens": pre["prefill_tokens"],
                "quant_append_us": round(pre["prefill_us"], 2),
                "quant_append_gbs": round(ach, 1), "quant_append_frac": round(ach / peak, 4),
                "roofline": {"bound": "hbm", "achieved": round(kach, 1), "peak": peak, "unit": "GB/s",
                             "frac": round(kach / peak, 4), "nominal_peak": NOMINAL_HBM_GBS,
                             "frac_of_nominal": round(kach / NOMINAL_HBM_GBS, 4),
                             "traffic": profiled_traffic("prefill_128k_prefix16", "prefill"),
                             "traffic_note": "lower bound: codes written back from L2 after the kernel ends "
                                             "are not counted in its DRAM bytes",
                             "kernel": "oscar_prefill_append_kernel",
                             "launch_us": round(pre["prefill_kernel_us"], 2),
                             "algorithmic_bytes_per_launch": pre["prefill_kernel_bytes"]},
                "prefix16_decode_us": round(pre["prefix_decode_us"], 2),
                "prefix16_shared_prefix_decode_us": round(pre["prefix_shared_decode_us"], 2),
                "prefix16_logical_gbs": round(pre["prefix_logical_bytes"] / (pre["prefix_decode_us"] * 1e-6) / 1e9, 1),
                "prefix16_unique_bytes": pre["prefix_unique_bytes"],
                "prefix16_logical_bytes": pre["prefix_logical_bytes"],
            }
        out["footprint"] = [footprint(n) for n in ("qwen3_32b_bs28_100k", "qwen3_8b_bs1_32k",
                                                   "qwen3_32b_bs28_100k_pages", "qwen3_8b_bs1_32k_pages")]
        # one flat object per further decode workload, last on the line, so a
        # reader that keeps only top-level scalars (or only the line's tail) still
        # has each workload's kernel time and roofline fraction
        short = {"qwen3_32b_bs28_100k": "bs28_100k", "qwen3_8b_bs16_ragged": "bs16_ragged",
                 "qwen3_32b_bs28_100k_pages": "bs28_100k_pages"}
        for r in extras:
            rf = roof(r)
            out[short.get(r["workload"], r["workload"])] = {
                "workload": r["workload"], "kernel_us": round(r["kernel_us"], 2),
                "kernel_gbs": rf["achieved"], "frac": rf["frac"], "frac_of_nominal": rf["frac_of_nominal"],
                "traffic": rf["traffic"], "kernel_bytes": r["kernel_bytes"],
                "decode_us": round(r["decode_us"], 2), "us_per_step": round(r["us_per_step"], 2),
                "sm_mhz": r["clocks"].get("sm_mhz"), "clock_reasons": ",".join(r["clocks"].get("reasons", []))}
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
