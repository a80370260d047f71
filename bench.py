"""Benchmark of the SWA + KV-sink hot path on one GB300 per rank.

Default workload (the headline line): the decode step at batch 64, 8 query /
2 KV heads, head_dim 64, 64 pinned sink slots + a full 256-slot ring with a
random ring offset, int8 group-32 K/V -- one step = fused quantise-and-append
of one new bf16 token per sequence + one decode over sink + ring.  Metric:
decode KV GB/s (algorithmic bytes: every live cache byte read once, plus q,
out and the appended token).  The other measured configurations (packed
prefill, compressed prefill, large-batch decode sweep) are timed in the same
run and reported under "rows".

Timing: W >= 3 untimed warm-up steps, then exactly K steps captured in a CUDA
graph and replayed between CUDA events on the launching stream, with a
barrier + synchronize on both sides (max over ranks).  Inputs smaller than
L2 rotate through enough replicas to total more than 4x L2, so every step reads
cold HBM.  Clocks are sampled with nvidia-smi during the timed region.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
METRIC = "SWA+sink attn prefill tok/s and decode KV GB/s (% of HBM/tensor roofline)"


# ----------------------------------------------------------------------------
# environment helpers
# ----------------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# workloads on the device (inputs generated on the host from seeds)
# ----------------------------------------------------------------------------

def dev_bf16(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def make_decode_state(torch, nd, B, Hq, Hkv, d, S, W, seed, replicas):
    """Replicas of a fully populated cache (quantised on the device from N(0,1)
    bf16 tokens with nd_kv_quant_rows), a bf16 query, and per-step new tokens."""
    from workloads import philox
    rng = philox(seed)
    reps = []
    ns = S + W
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    for r in range(replicas):
        cache = nd.KVCache.empty(B, Hkv, d, S, W)
        for codes, scales in ((cache.k_codes, cache.k_scale), (cache.v_codes, cache.v_scale)):
            x = torch.randn((B, Hkv, ns, d), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
            nd.nd_kv_quant_rows(x, codes, scales)
            del x
        start = rng.integers(0, W, size=B).astype(np.int32)
        cache.sink_len.fill_(S)
        cache.ring_len.fill_(W)
        cache.ring_start.copy_(torch.from_numpy(start))
        cache.seq_len.copy_(torch.from_numpy((S + W + start).astype(np.int32)))
        q = torch.randn((B, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
        kn = torch.randn((B, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn((B, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
        out = torch.empty_like(q)
        reps.append(dict(cache=cache, q=q, kn=kn, vn=vn, out=out))
    nbytes = nd.nd_swa_sink_decode_workspace_size(B, Hq, Hkv, d, S + W)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    return reps, ws


def decode_bytes(B, Hq, Hkv, d, S, W):
    cache = B * (S + W) * Hkv * (2 * d + 2 * (d // 32) * 4)
    qo = 2 * B * Hq * d * 2
    append = B * Hkv * (2 * d * 2 + 2 * d + 2 * (d // 32) * 4)
    return cache, qo, append


def visible_pairs_packed(seg, sink, W):
    """Visible (q, k) pairs per batch row for contiguous segments that open
    with a sink prefix (the packed workload's layout): row i of a segment sees
    min(i+1, W) window keys plus the sink keys that lie before its window."""
    total = []
    for b in range(seg.shape[0]):
        n = 0
        s = 0
        T = seg.shape[1]
        while s < T:
            e = s
            while e < T and seg[b, e] == seg[b, s]:
                e += 1
            if seg[b, s] > 0:
                ns = int(sink[b, s:e].sum())
                i = np.arange(e - s)
                win = np.minimum(i + 1, W)
                extra = np.clip(np.minimum(ns, i - W + 1), 0, None)
                n += int(win.sum() + extra.sum())
            s = e
        total.append(n)
    return np.array(total)


def performed_tiles_packed(seg, sink, W, span=128, bn=64):
    """(128-row span, 64-key tile) pairs the prefill kernel computes, summed
    over batch rows: the tile plan's rule -- the tile holds a key whose segment
    id lies in the span's id range, and it reaches into the span's window or
    holds a sink."""
    B, T = seg.shape
    n_kt = (T + bn - 1) // bn
    total = 0
    for b in range(B):
        s = np.where(seg[b] > 0, seg[b], 0)
        pad = np.zeros(n_kt * bn, np.int64)
        pad[:T] = s
        tiles = pad.reshape(n_kt, bn)
        big = np.iinfo(np.int64).max
        lo = np.where(tiles > 0, tiles, big).min(axis=1)
        hi = tiles.max(axis=1)
        skp = np.zeros(n_kt * bn, bool)
        skp[:T] = sink[b] != 0
        any_sink = skp.reshape(n_kt, bn).any(axis=1)
        for q0 in range(0, T, span):
            q1 = min(T, q0 + span) - 1
            qs = s[q0:q1 + 1]
            qs = qs[qs > 0]
            if qs.size == 0:
                continue
            j = np.arange(q1 // bn + 1)
            ok = (lo[j] <= hi[j]) & (lo[j] <= qs.max()) & (hi[j] >= qs.min())
            in_win = (W == 0) | ((j + 1) * bn - 1 >= q0 - W + 1)
            total += int((ok & (in_win | any_sink[j])).sum())
    return total


def performed_tiles_compressed(T, W, block, span=128, bn=64):
    """The same count for one compressed-attention row: pooled tiles below the
    block threshold plus exact tiles reaching into the window."""
    total = 0
    nb = T // block
    for q0 in range(0, T, span):
        q1 = min(T, q0 + span) - 1
        lim = q1 - W + 1
        ncol = min(lim // block, nb) if lim >= block else 0
        total += (ncol + bn - 1) // bn
        j = np.arange(q1 // bn + 1)
        total += int(((j + 1) * bn - 1 >= q0 - W + 1).sum())
    return total


def visible_pairs_compressed(T, W, b):
    q = np.arange(T)
    exact = np.minimum(q + 1, W)
    pooled = np.clip((q - W + 1) // b, 0, T // b)
    return int(exact.sum() + pooled.sum())


# ----------------------------------------------------------------------------
# timing
# ----------------------------------------------------------------------------

def time_graph(torch, fn_step, steps, warmup, dist=None):
    """Warm up `warmup` steps eagerly, capture exactly `steps` steps in a CUDA
    graph, replay it once between events; returns ms for the K steps (max
    over ranks)."""
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn_step(i)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            fn_step(i)
    # one untimed replay brings the graph's own launch path up
    graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    with torch.cuda.stream(stream):
        graph.replay()
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    return max_over_ranks(torch, ms, dist, "cuda")


def max_over_ranks(torch, ms, dist, device):
    """The slowest rank's time: every rank's work counts only once all ranks
    are done."""
    if not dist:
        return ms
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: independent sequences)."""
    return base + 7919 * rank


def job_throughput(bytes_per_step_per_rank, steps, world, ms_max):
    """Whole-job GB/s: bytes all ranks processed / the slowest rank's time."""
    return bytes_per_step_per_rank * steps * world / (ms_max * 1e-3) / 1e9


# ----------------------------------------------------------------------------
# the measured rows
# ----------------------------------------------------------------------------

def bench_decode(torch, nd, B, Hq, Hkv, d, S, W, steps, warmup, seed, pk, dist=None, with_append=True):
    cache_b, qo_b, app_b = decode_bytes(B, Hq, Hkv, d, S, W)
    per_rep = cache_b + qo_b + app_b
    replicas = max(1, math.ceil(4 * L2_BYTES / per_rep))
    reps, ws = make_decode_state(torch, nd, B, Hq, Hkv, d, S, W, seed, replicas)

    def step(i):
        r = reps[i % replicas]
        if with_append:   # one decode step: append the current token, attend with it
            nd.nd_swa_sink_decode_step(r["q"], r["cache"], r["kn"], r["vn"], W, out=r["out"], workspace=ws)
        else:
            nd.nd_swa_sink_decode(r["q"], r["cache"], W, out=r["out"], workspace=ws)

    def decode_only(i):
        r = reps[i % replicas]
        nd.nd_swa_sink_decode(r["q"], r["cache"], W, out=r["out"], workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    ms_kernel = time_graph(torch, decode_only, steps, warmup, dist)
    step_bytes = cache_b + qo_b + (app_b if with_append else 0)
    split = nd.nd_swa_sink_decode_workspace_size(B, Hq, Hkv, d, S + W) > 0
    # unsplit with at most 4 KV heads, a sequence's CTAs form one small cluster
    # and the step is a single fused launch (the library's rule); otherwise the
    # append is its own launch and a split decode adds its combine launch
    fused = with_append and not split and Hkv <= 4
    launches_per_step = 1 if fused else (1 if with_append else 0) + (2 if split else 1)
    step_gbs = step_bytes / (ms / steps * 1e-3) / 1e9
    decode_gbs = (cache_b + qo_b) / (ms_kernel / steps * 1e-3) / 1e9
    if fused:   # the dominant (only) kernel of the step is the fused one
        kernel = dict(name="decode_kernel (nd_swa_sink_decode_step: fused append + decode)",
                      ms_per_launch=ms / steps, bytes_per_launch=step_bytes, gbs=step_gbs, frac=step_gbs / pk["hbm"])
    else:
        kernel = dict(name="decode_kernel (nd_swa_sink_decode)", ms_per_launch=ms_kernel / steps,
                      bytes_per_launch=cache_b + qo_b, gbs=decode_gbs, frac=decode_gbs / pk["hbm"])
    kernel["decode_only"] = dict(ms_per_launch=ms_kernel / steps, bytes_per_launch=cache_b + qo_b, gbs=decode_gbs)
    return dict(
        ms_per_step=ms / steps, gbs=step_gbs, bytes_per_step=step_bytes,
        replicas=replicas, launches=launches_per_step * steps, kernel=kernel, _state=(reps, ws))


def bench_packed_prefill(torch, nd, steps, warmup, pk, dist=None, batch=8, cpu_budget=None):
    from workloads import packed_prefill
    w = packed_prefill(B=batch)
    B, T, Hq, d = w["q"].shape
    Hkv = w["k"].shape[2]
    q, k, v = dev_bf16(torch, w["q_bits"]), dev_bf16(torch, w["k_bits"]), dev_bf16(torch, w["v_bits"])
    seg = torch.from_numpy(w["seg_ids"]).cuda()
    sink = torch.from_numpy(w["sink"]).cuda()
    out = torch.empty_like(q)
    nbytes = nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, Hq, Hkv, d, w["rope_theta"], 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")

    def step(i):
        nd.nd_swa_sink_prefill(q, k, v, seg, sink, w["window"], rope_theta=w["rope_theta"], out=out, workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    # the attention kernel's share: the same call on pre-rotated q/k (no RoPE pass)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    nd.nd_rope_apply(q, qr, w["rope_theta"])
    nd.nd_rope_apply(k, kr, w["rope_theta"])
    ws0 = torch.empty(max(nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, Hq, Hkv, d, 0.0, 0), 16),
                      dtype=torch.uint8, device="cuda")

    def attn(i):
        nd.nd_swa_sink_prefill(qr, kr, v, seg, sink, w["window"], rope_theta=0.0, out=out, workspace=ws0)

    ms_attn = time_graph(torch, attn, steps, warmup, dist)
    pairs = int(visible_pairs_packed(w["seg_ids"], w["sink"], w["window"]).sum())
    flops = 4.0 * d * pairs * Hq
    tiles = performed_tiles_packed(w["seg_ids"], w["sink"], w["window"])
    tile_flops = 4.0 * 128 * 64 * d * tiles * Hq
    t, ta = ms / steps * 1e-3, ms_attn / steps * 1e-3
    oracle_row = None
    if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
        try:
            oracle_row = oracle_prefill_sample("packed", w, 4, 1, cpu_budget)
        except Exception as ex:  # the product path never depends on it
            oracle_row = {"tok_s": None, "sample": f"unavailable: {ex}"}
    return dict(config=f"packed prefill B{B} T{T} Hq{Hq} Hkv{Hkv} d{d} W256 RoPE, 3-6 segments with 64-512 sink prefixes",
                oracle=oracle_row,
                ms_per_step=ms / steps, tok_s=B * T / t, tflops=flops / t / 1e12,
                frac=flops / t / 1e12 / pk["bf16"], visible_pairs=pairs, flops_per_step=flops,
                attn_ms=ms_attn / steps, tiles=tiles * Hq, tile_flops=tile_flops,
                tile_tflops=tile_flops / ta / 1e12, tile_frac=tile_flops / ta / 1e12 / pk["bf16"],
                launches=4 * steps)


def bench_compressed(torch, nd, steps, warmup, pk, dist=None, cpu_budget=None):
    from workloads import compressed
    w = compressed()
    B, T, H, d = w["q"].shape
    q, k, v = dev_bf16(torch, w["q_bits"]), dev_bf16(torch, w["k_bits"]), dev_bf16(torch, w["v_bits"])
    nb = T // w["block"]
    pkk = torch.empty((B, nb, H, d), dtype=torch.bfloat16, device="cuda")
    pvv = torch.empty_like(pkk)
    out = torch.empty_like(q)
    nbytes = nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, H, H, d, w["rope_theta"], w["block"])
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")

    def step(i):
        nd.nd_kv_compress_pool(k, v, w["block"], w["rope_theta"], pooled_k=pkk, pooled_v=pvv)
        nd.nd_swa_sink_prefill(q, k, v, None, None, w["window"], rope_theta=w["rope_theta"], pooled_k=pkk,
                               pooled_v=pvv, block=w["block"], out=out, workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    nd.nd_rope_apply(q, qr, w["rope_theta"])
    nd.nd_rope_apply(k, kr, w["rope_theta"])
    ws0 = torch.empty(max(nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, H, H, d, 0.0, w["block"]), 16),
                      dtype=torch.uint8, device="cuda")

    def attn(i):
        nd.nd_swa_sink_prefill(qr, kr, v, None, None, w["window"], rope_theta=0.0, pooled_k=pkk, pooled_v=pvv,
                               block=w["block"], out=out, workspace=ws0)

    ms_attn = time_graph(torch, attn, steps, warmup, dist)
    pairs = visible_pairs_compressed(T, w["window"], w["block"]) * B * H
    flops = 4.0 * d * pairs
    tiles = performed_tiles_compressed(T, w["window"], w["block"]) * B * H
    tile_flops = 4.0 * 128 * 64 * d * tiles
    t, ta = ms / steps * 1e-3, ms_attn / steps * 1e-3
    oracle_row = None
    if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
        try:
            oracle_row = oracle_prefill_sample("compressed", w, 2, 2, cpu_budget)
        except Exception as ex:  # the product path never depends on it
            oracle_row = {"tok_s": None, "sample": f"unavailable: {ex}"}
    return dict(config="compressed prefill B4 T4096 H16 d64 W256 b4 RoPE", oracle=oracle_row,
                ms_per_step=ms / steps,
                tok_s=B * T / t, tflops=flops / t / 1e12, frac=flops / t / 1e12 / pk["bf16"],
                visible_pairs=pairs, attn_ms=ms_attn / steps, tiles=tiles, tile_flops=tile_flops,
                tile_tflops=tile_flops / ta / 1e12, tile_frac=tile_flops / ta / 1e12 / pk["bf16"],
                launches=5 * steps)


# ----------------------------------------------------------------------------
# e2e and CPU baseline
# ----------------------------------------------------------------------------

def e2e_decode(torch, nd, state, B, Hq, Hkv, d, S, W, steps, warmup):
    """Same step through the public API with host buffers: one
    nd_swa_sink_decode_step_host_packed call per step, which enqueues the
    pinned host -> device copy of the step's query and new token, the append +
    decode and the device -> host copy of the output; all inside the timed
    region."""
    reps, _ = state
    r = reps[0]
    # each step's inputs in one page-locked allocation (q | k_new | v_new)
    # and its output in another, through the packed form of the call: one
    # copy each way.  The per-step tensors exist before the timed region, as
    # a serving loop's buffers would.
    nq, nk = B * Hq * d, B * Hkv * d
    ins, outs = [], []
    for _ in range(steps + warmup):
        t_ = torch.empty(nq + 2 * nk, dtype=torch.bfloat16).pin_memory()
        t_.copy_(torch.randn(nq + 2 * nk).to(torch.bfloat16))
        ins.append(t_)
        outs.append(torch.empty((B, Hq, d), dtype=torch.bfloat16).pin_memory())
    stream = torch.cuda.current_stream()
    ws = torch.empty(nd.nd_swa_sink_decode_step_host_workspace_size(B, Hq, Hkv, d, S + W),
                     dtype=torch.uint8, device="cuda")
    st = r["cache"].struct()
    cache = r["cache"]

    def one(i):
        nd.nd_swa_sink_decode_step_host_packed(ins[i], cache, Hq, W, outs[i], workspace=ws, stream=stream,
                                               cache_struct=st)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    t0 = time.perf_counter()
    for i in range(steps):
        one(warmup + i)
    host_s = time.perf_counter() - t0
    e.record(stream)
    e.synchronize()
    ms = s.elapsed_time(e)
    cache_b, qo_b, app_b = decode_bytes(B, Hq, Hkv, d, S, W)
    h2d = B * Hq * d * 2 + 2 * B * Hkv * d * 2
    d2h = B * Hq * d * 2
    return dict(value=(cache_b + qo_b + app_b) / (ms / steps * 1e-3) / 1e9, unit="GB/s",
                h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h, ms_per_step=ms / steps,
                host_enqueue_ms_per_step=host_s * 1e3 / steps)


def oracle_prefill_sample(kind, w, heads, kv_heads, budget_s):
    """Times the oracle's prefill on the host beside a prefill row: one
    sequence of the row's workload with its first `heads` query heads (and
    their `kv_heads` KV heads), repeated until budget_s elapses (at least
    once); tok/s scaled to the whole row: tokens x heads/Hq per run time."""
    import oracle
    B, T, Hq, d = w["q"].shape
    q, k, v = w["q"][:1, :, :heads], w["k"][:1, :, :kv_heads], w["v"][:1, :, :kv_heads]
    n, t0 = 0, time.perf_counter()
    while True:
        if kind == "packed":
            oracle.swa_sink_prefill(q, k, v, w["seg_ids"][:1], w["sink"][:1], w["window"], w["rope_theta"])
        else:
            oracle.compressed_prefill(q, k, v, w["window"], w["block"], w["rope_theta"])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return dict(tok_s=T * heads / Hq * n / el, cores=min(oracle.num_threads(), heads * T), kind="oracle",
                sample=f"{n} run(s) of one sequence (T{T}) x {heads} of {Hq} query heads in {el:.1f} s "
                       f"(fp64 dense oracle, OpenMP over rows and heads), scaled by heads to the row")


def oracle_decode_sample(B, Hq, Hkv, d, S, W, seed, budget_s):
    """Times the oracle's decode on the host: the same workload, one full step
    (every sequence) per iteration, repeated until budget_s elapses."""
    import oracle
    from workloads import decode_cache
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=seed, full=True)
    ref = oracle.Cache(B, Hkv, d, S, W)
    ref.k_codes[...], ref.k_scale[...] = oracle.quant_g32(w["k"])
    ref.v_codes[...], ref.v_scale[...] = oracle.quant_g32(w["v"])
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        getattr(ref, f)[...] = w[f]
    cache_b, qo_b, _ = decode_bytes(B, Hq, Hkv, d, S, W)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(w["q"], ref, W)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    threads = min(oracle.num_threads(), Hq)   # the oracle parallelises over query heads
    return dict(value=(cache_b + qo_b) * n / el / 1e9, unit="GB/s", cores=threads, kind="oracle",
                sample=f"{n} full decode steps of the B{B} Hq{Hq} Hkv{Hkv} d{d} S{S}+W{W} workload in {el:.1f} s "
                       f"(fp64 dense oracle, OpenMP over query heads)", seconds=el)


# ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nd", choices=["nd", "reference"])
    ap.add_argument("--rows", default="all", help="comma list of extra rows: sweep,packed,compressed or none")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--sweep-batches", default="32,64,128,256,512",
                    help="batch sizes of the large-batch decode sweep (all five = the measured configuration)")
    ap.add_argument("--packed-batch", type=int, default=8,
                    help="sequences in the packed-prefill row (8 = the measured configuration; smaller for profiling)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    B, Hq, Hkv, d, S, W = 64, 8, 2, 64, 64, 256
    workload = "decode step B64 Hq8 Hkv2 d64, 64 sink slots + 256-slot ring (full, random offset), int8 g32 K/V"

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        per_step = []
        for i in range(warmup + steps):
            r = oracle_decode_sample(B, Hq, Hkv, d, S, W, 1234 + 1, budget_s=0.0)
            if i >= warmup:
                per_step.append(r["seconds"])
        ms = 1e3 * sum(per_step) / len(per_step)
        cache_b, qo_b, _ = decode_bytes(B, Hq, Hkv, d, S, W)
        val = (cache_b + qo_b) / (ms * 1e-3) / 1e9
        line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus, "steps": steps,
                "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": {"workload": workload, "l2": "host run"},
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": "each step is one full decode step of the workload on the fp64 oracle"},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)
    import sliding_window_kv_swa_gb300 as nd
    pk = peaks()
    dev_index = torch.cuda.current_device()

    with ClockSampler(dev_index) as clk:
        head = bench_decode(torch, nd, B, Hq, Hkv, d, S, W, steps, warmup, seed=rank_seed(1234 + 1, rank), pk=pk,
                            dist=dist)
    clocks = clk.summary()
    e2e = e2e_decode(torch, nd, head.pop("_state"), B, Hq, Hkv, d, S, W, min(steps, 200), warmup)

    rows = {}
    want = set(args.rows.split(",")) if args.rows not in ("all", "none") else (
        {"sweep", "packed", "compressed"} if args.rows == "all" else set())
    if "sweep" in want:
        sweep = {}
        for Bs in [int(x) for x in args.sweep_batches.split(",")]:
            r = bench_decode(torch, nd, Bs, 32, 8, 128, 1024, 256, max(20, steps // 4), warmup,
                             seed=rank_seed(1234 + 4, rank), pk=pk, dist=dist)
            r.pop("_state")
            sweep[f"B{Bs}"] = dict(gbs=r["gbs"], frac=r["gbs"] / pk["hbm"], ms_per_step=r["ms_per_step"],
                                  kernel_gbs=r["kernel"]["gbs"], kernel_frac=r["kernel"]["frac"])
            torch.cuda.empty_cache()
        rows["decode_sweep"] = dict(config="decode + fused append, Hq32 Hkv8 d128, 1024 sinks + 256 ring", **sweep)
    if "packed" in want:
        rows["packed_prefill"] = bench_packed_prefill(torch, nd, max(10, steps // 10), warmup, pk, dist,
                                                      batch=args.packed_batch,
                                                      cpu_budget=min(5.0, args.cpu_budget))
        torch.cuda.empty_cache()
    if "compressed" in want:
        rows["compressed_prefill"] = bench_compressed(torch, nd, max(10, steps // 10), warmup, pk, dist,
                                                      cpu_budget=min(5.0, args.cpu_budget))
        torch.cuda.empty_cache()

    value = job_throughput(head["bytes_per_step"], steps, world, head["ms_per_step"] * steps)
    k = head["kernel"]
    traffic = None
    try:
        tr = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        traffic = tr.get("decode_step@decode_b64") if "fused" in k["name"] else tr.get("decode@decode_b64")
    except Exception:
        pass
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 KV / bf16 q,out / fp32 accum", "data": "synthetic",
        "config": {"workload": workload, "l2": f"rotating {head['replicas']} cache replicas (> 4x L2)",
                   "timing": "CUDA graph of K steps, CUDA events"},
        "roofline": {"bound": "hbm", "achieved": k["gbs"], "peak": pk["hbm"], "unit": "GB/s", "frac": k["frac"],
                     "traffic": traffic, "kernel": k["name"], "peak_source": pk["src"],
                     "ms_per_launch": k["ms_per_launch"], "bytes_per_launch": k["bytes_per_launch"]},
        "gpu_launches": head["launches"],
        "clocks": clocks,
        "e2e": e2e,
        "rows": rows,
    }
    if rank == 0:
        try:
            line["cpu_baseline"] = oracle_decode_sample(B, Hq, Hkv, d, S, W, 1234 + 1, args.cpu_budget)
            line["cpu_baseline"].pop("seconds", None)
        except Exception as ex:  # the product path never depends on it
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 0, "kind": "oracle",
                                    "sample": f"unavailable: {ex}"}
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
