"""Benchmark of the SWA + KV-sink hot path on one GB300 per rank.

Headline (`value`): the decode step of the large-batch configuration at its
largest batch -- B512, 32 query / 8 KV heads, head_dim 128, 1024 pinned sink
slots + a full 256-slot ring with a random ring offset, int8 group-32 K/V; one
step = quantise-and-append of one new bf16 token per sequence + one decode
over sink + ring.  Metric: decode KV GB/s (algorithmic bytes: every live cache
byte read once, plus q, out and the appended token).  `roofline` is the
decode kernel alone on the same cache.  Every other measured configuration
is a row under "rows" with its own roofline and oracle figure: the B64 decode
step, the rest of the batch sweep, a window sweep, packed and compressed
prefill (block 4 and 8), fp32 tiny prefill, block pooling, the standalone
append, the prefill->cache handoff and the compressed-attention decode step.

Timing: W >= 3 untimed warm-up steps, then exactly K steps captured in a CUDA
graph and replayed between CUDA events on the launching stream, with a
barrier + synchronize on both sides (max over ranks).  Inputs smaller than
4x L2 rotate through enough replicas to total more than that, so every step
reads cold HBM.  Clocks are sampled with nvidia-smi during the headline's
timed region.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (a bounded sample of its sequences per step).
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
# rooflines
# ----------------------------------------------------------------------------

def roofline(bound, work, ms, peak, unit, kernel, peak_source, traffic=None):
    """Roofline record of one kernel: `work` algorithmic bytes (GB/s) or
    flops (TFLOP/s) per launch over its measured time per launch."""
    scale = 1e9 if unit == "GB/s" else 1e12
    achieved = work / (ms * 1e-3) / scale
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": traffic, "kernel": kernel, "ms_per_launch": ms, "work_per_launch": work,
            "peak_source": peak_source}


def alu_fp32_peak_tflops():
    """fp32 FFMA peak: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def load_traffic(key):
    try:
        return json.load(open(os.path.join(ROOT, "profiles", "traffic.json"))).get(key)
    except Exception:
        return None


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

def bench_decode(torch, nd, B, Hq, Hkv, d, S, W, steps, warmup, seed, pk, dist=None, traffic_key=None):
    """Decode step (append the current token, attend with it) and the decode
    kernel alone, on rotating cache replicas."""
    cache_b, qo_b, app_b = decode_bytes(B, Hq, Hkv, d, S, W)
    per_rep = cache_b + qo_b + app_b
    replicas = max(1, math.ceil(4 * L2_BYTES / per_rep))
    reps, ws = make_decode_state(torch, nd, B, Hq, Hkv, d, S, W, seed, replicas)

    def step(i):
        r = reps[i % replicas]
        nd.nd_swa_sink_decode_step(r["q"], r["cache"], r["kn"], r["vn"], W, out=r["out"], workspace=ws)

    def decode_only(i):
        r = reps[i % replicas]
        nd.nd_swa_sink_decode(r["q"], r["cache"], W, out=r["out"], workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    ms_kernel = time_graph(torch, decode_only, steps, warmup, dist)
    step_bytes = cache_b + qo_b + app_b
    split = nd.nd_swa_sink_decode_workspace_size(B, Hq, Hkv, d, S + W) > 0
    # unsplit with at most 4 KV heads, a sequence's CTAs form one small cluster
    # and the step is a single fused launch (the library's rule); otherwise the
    # append is its own launch and a split decode adds its combine launch
    fused = not split and Hkv <= 4
    launches_per_step = 1 if fused else 1 + (2 if split else 1)
    t, tk = ms / steps, ms_kernel / steps
    if fused:   # the step's only kernel is the fused one
        rl = roofline("hbm", step_bytes, t, pk["hbm"], "GB/s",
                      "decode_kernel (nd_swa_sink_decode_step: fused append + decode)", pk["src"],
                      load_traffic(traffic_key))
    else:
        rl = roofline("hbm", cache_b + qo_b, tk, pk["hbm"], "GB/s", "decode_kernel (nd_swa_sink_decode)", pk["src"],
                      load_traffic(traffic_key))
    return dict(config=f"decode step B{B} Hq{Hq} Hkv{Hkv} d{d}, {S} sink slots + {W}-slot ring (full), "
                       f"int8 g32 K/V, append of one bf16 token per sequence",
                ms_per_step=t, gbs=step_bytes / (t * 1e-3) / 1e9, frac=step_bytes / (t * 1e-3) / 1e9 / pk["hbm"],
                bytes_per_step=step_bytes, decode_kernel_ms=tk,
                decode_kernel_gbs=(cache_b + qo_b) / (tk * 1e-3) / 1e9,
                decode_kernel_frac=(cache_b + qo_b) / (tk * 1e-3) / 1e9 / pk["hbm"],
                replicas=replicas, launches=launches_per_step * steps, fused=fused, roofline=rl,
                _state=(reps, ws))


def e2e_decode(torch, nd, state, B, Hq, Hkv, d, S, W, steps, warmup, n_buffers=8):
    """The same step through the public API with host buffers: one
    nd_swa_sink_decode_step_host_packed call per step on page-locked host
    memory.  The step's kernels read the query and new token and write the
    output over the host link in place, so every input and output byte
    crosses it inside the timed region.  The steps walk the same cache
    replicas as the timed step."""
    reps, _ = state
    nq, nk = B * Hq * d, B * Hkv * d
    ins, outs = [], []
    for _ in range(n_buffers):   # a serving loop's reusable page-locked buffers
        t_ = torch.empty(nq + 2 * nk, dtype=torch.bfloat16).pin_memory()
        t_.copy_(torch.randn(nq + 2 * nk).to(torch.bfloat16))
        ins.append(t_)
        outs.append(torch.empty((B, Hq, d), dtype=torch.bfloat16).pin_memory())
    stream = torch.cuda.current_stream()
    ws = torch.empty(nd.nd_swa_sink_decode_step_host_workspace_size(B, Hq, Hkv, d, S + W),
                     dtype=torch.uint8, device="cuda")
    structs = [r["cache"].struct() for r in reps]

    def one(i):
        r = i % len(reps)
        nd.nd_swa_sink_decode_step_host_packed(ins[i % n_buffers], reps[r]["cache"], Hq, W, outs[i % n_buffers],
                                               workspace=ws, stream=stream, cache_struct=structs[r])

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
                host_enqueue_ms_per_step=host_s * 1e3 / steps, cache_replicas=len(reps))


def bench_compressed_decode(torch, nd, steps, warmup, pk, dist=None, B=128, H=16, d=64, T=4096, W=256, block=4):
    """Compressed-attention decode step at a 4096-token context: 960 visible
    pooled blocks + 256 exact keys per sequence (random int8 contents),
    rotating replicas."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + 7)
    n_steps = warmup + steps + 1
    n_vis0 = (T - W + 1) // block
    sink_cap = (T + n_steps) // block + 1    # every block the run closes fits
    vis_mid = (T + n_steps // 2 - W + 1) // block
    per_step = B * H * ((vis_mid + W) * (2 * d + 2 * (d // 32) * 4)) + 2 * B * H * d * 2 + B * H * (2 * d * 2)
    replicas = max(1, math.ceil(4 * L2_BYTES / (B * H * (sink_cap + W) * (2 * d + 2 * (d // 32) * 4))))
    reps = []
    for _ in range(replicas):
        # codes uniform in [-127, 127] and scales in the absmax/127 range of
        # N(0,1) groups, drawn on the device
        ns = sink_cap + W
        codes = lambda: torch.randint(-127, 128, (B, H, ns, d), generator=g, device="cuda").to(torch.int8)
        scales = lambda: torch.rand((B, H, ns, d // 32), generator=g, device="cuda") * (1.1 / 127) + 2.2 / 127
        kv = nd.KVCache(codes(), codes(), scales(), scales(),
                        torch.full((B,), n_vis0, dtype=torch.int32, device="cuda"),
                        torch.randint(0, W, (B,), generator=g, device="cuda").to(torch.int32),
                        torch.full((B,), W, dtype=torch.int32, device="cuda"),
                        torch.full((B,), T, dtype=torch.int32, device="cuda"), sink_cap, W)
        cache = nd.CompressedCache(kv, torch.zeros((B, H, d), device="cuda"), torch.zeros((B, H, d), device="cuda"),
                                   block, 0)
        q = torch.randn((B, H, d), device="cuda").to(torch.bfloat16)
        kn = torch.randn((B, H, d), device="cuda").to(torch.bfloat16)
        vn = torch.randn((B, H, d), device="cuda").to(torch.bfloat16)
        reps.append(dict(cache=cache, st=cache.struct(), q=q, kn=kn, vn=vn, out=torch.empty_like(q)))
    ws = torch.empty(nd.nd_compressed_decode_step_workspace_size(B, H, H, d, sink_cap + W), dtype=torch.uint8,
                     device="cuda")

    def step(i):
        r = reps[i % replicas]
        nd.nd_compressed_decode_step(r["q"], r["cache"], r["kn"], r["vn"], W, 10000.0, out=r["out"], workspace=ws,
                                     cache_struct=r["st"])

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    split = nd.nd_swa_sink_decode_workspace_size(B, H, H, d, sink_cap + W) > 0
    return dict(config=f"compressed-attention decode step B{B} H{H} (MHA) d{d}, context {T}: {n_vis0}+ visible "
                       f"pooled blocks (b{block}) + {W} exact keys, int8 g32, RoPE; append + incremental pooling",
                ms_per_step=t, bytes_per_step=per_step, replicas=replicas, launches=(3 if split else 2) * steps,
                roofline=roofline("hbm", per_step, t, pk["hbm"], "GB/s",
                                  "compressed_append_kernel + decode_kernel (whole step)", pk["src"],
                                  load_traffic(f"compressed_decode@b{B}")))


def bench_window_sweep(torch, nd, steps, warmup, pk, dist, windows=(160, 256, 512, 1024), B=128):
    """The decode step at the windows effective_kv_window can return (multiples
    of 32, at least 160): the cost follows sinks + window."""
    out = {}
    for W in windows:
        r = bench_decode(torch, nd, B, 32, 8, 128, 1024, W, steps, warmup, seed=1234 + 8, pk=pk, dist=dist)
        r.pop("_state")
        out[f"W{W}"] = dict(ms_per_step=r["ms_per_step"], gbs=r["gbs"], frac=r["frac"], roofline=r["roofline"])
        torch.cuda.empty_cache()
    return dict(config=f"decode step B{B} Hq32 Hkv8 d128, 1024 sinks + a full ring of W slots", **out)


# ----------------------------------------------------------------------------
# prefill
# ----------------------------------------------------------------------------

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
    tiles = nd.nd_swa_sink_prefill_tiles(ws0, B, T, Hq, Hkv, d, 0.0, 0)   # what the kernel's plan performed
    pairs = int(visible_pairs_packed(w["seg_ids"], w["sink"], w["window"]).sum())
    flops = 4.0 * d * pairs * Hq
    tile_flops = 4.0 * 128 * 64 * d * tiles
    t, ta = ms / steps, ms_attn / steps
    oracle_row = None
    if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
        try:
            oracle_row = oracle_prefill_sample("packed", w, 4, 1, cpu_budget)
        except Exception as ex:  # the product path never depends on it
            oracle_row = {"tok_s": None, "sample": f"unavailable: {ex}"}
    return dict(config=f"packed prefill B{B} T{T} Hq{Hq} Hkv{Hkv} d{d} W256 RoPE, 3-6 segments with 64-512 sink prefixes",
                oracle=oracle_row, ms_per_step=t, tok_s=B * T / (t * 1e-3), step_tflops=flops / (t * 1e-3) / 1e12,
                visible_pairs=pairs, flops_per_step=flops, attn_ms=ta,
                attn_algorithmic=roofline("tensor", flops, ta, pk["bf16"], "TFLOP/s",
                                          "prefill_tc_kernel (visible pairs)", pk["src"]),
                tiles=tiles, tile_flops=tile_flops, tile_overhead=tile_flops / flops,
                roofline=roofline("tensor", tile_flops, ta, pk["bf16"], "TFLOP/s",
                                  "prefill_tc_kernel (tiles its plan performed)", pk["src"],
                                  load_traffic("prefill_tc@packed")),
                launches=4 * steps)


def bench_chunk(torch, nd, steps, warmup, pk, dist=None, B=8, Tc=4096, Hq=32, Hkv=8, d=128, S=1024, W=256,
                cpu_budget=None):
    """Chunked prefill of Tc new tokens per sequence against the large-batch
    cache layout (full sinks and ring, random int8 contents), then the
    chunk's append.  The cache advances with every call; its ring stays
    full, so every call does the same work."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + 9)
    ns = S + W
    codes = lambda: torch.randint(-127, 128, (B, Hkv, ns, d), generator=g, device="cuda").to(torch.int8)
    scales = lambda: torch.rand((B, Hkv, ns, d // 32), generator=g, device="cuda") * (1.1 / 127) + 2.2 / 127
    cache = nd.KVCache(codes(), codes(), scales(), scales(), torch.full((B,), S, dtype=torch.int32, device="cuda"),
                       torch.randint(0, W, (B,), generator=g, device="cuda").to(torch.int32),
                       torch.full((B,), W, dtype=torch.int32, device="cuda"),
                       torch.full((B,), S + W, dtype=torch.int32, device="cuda"), S, W)
    q = torch.randn((B, Tc, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Tc, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Tc, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    ws = torch.empty(nd.nd_swa_sink_chunk_prefill_workspace_size(B, Tc, Hq, Hkv, d, S, W, W), dtype=torch.uint8,
                     device="cuda")

    def step(i):
        nd.nd_swa_sink_chunk_prefill(q, k, v, cache, W, out=out, workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    tiles = nd.nd_swa_sink_chunk_prefill_tiles(ws, B, Tc, Hq, Hkv, d, S, W, W)
    # every chunk row sees the S sinks and W window keys (cache ring + chunk)
    pairs = B * Tc * (S + W)
    flops = 4.0 * d * pairs * Hq
    tile_flops = 4.0 * 128 * 64 * d * tiles
    orow = None
    if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
        try:
            orow = oracle_chunk_sample(Hq, Hkv, d, S, W, Tc, cpu_budget)
        except Exception as ex:  # the product path never depends on it
            orow = {"tok_s": None, "sample": f"unavailable: {ex}"}
    return dict(config=f"chunked prefill B{B} x {Tc} new tokens, Hq{Hq} Hkv{Hkv} d{d}, against {S} sinks + {W} ring "
                       f"(int8 g32), W{W}; gather + plan + attention + append", oracle=orow,
                ms_per_step=t, tok_s=B * Tc / (t * 1e-3), visible_pairs=pairs, tiles=tiles,
                tile_overhead=tile_flops / flops,
                algorithmic=roofline("tensor", flops, t, pk["bf16"], "TFLOP/s", "whole call (visible pairs)",
                                     pk["src"]),
                roofline=roofline("tensor", tile_flops, t, pk["bf16"], "TFLOP/s",
                                  "whole call (tiles the attention kernel's plan performed)", pk["src"],
                                  load_traffic(f"chunk_prefill@b{B}")),
                launches=4 * steps)


def oracle_chunk_sample(Hq, Hkv, d, S, W, Tc, budget_s, rows=256):
    """Times the oracle's chunked prefill on one sequence with the first
    `rows` tokens of a chunk, scaled to tok/s."""
    import oracle
    from workloads import philox, random_codes
    rng = philox(1234 + 9)
    kc, ks, vc, vs = random_codes(rng, 1, Hkv, S + W, d)
    ref = oracle.Cache(1, Hkv, d, S, W)
    ref.k_codes[...], ref.k_scale[...], ref.v_codes[...], ref.v_scale[...] = kc, ks, vc, vs
    ref.sink_len[:], ref.ring_len[:], ref.seq_len[:] = S, W, S + W
    q = rng.standard_normal((1, rows, Hq, d))
    k = rng.standard_normal((1, rows, Hkv, d))
    v = rng.standard_normal((1, rows, Hkv, d))
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.chunk_prefill(q, k, v, ref, W)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return dict(tok_s=rows * n / el, cores=oracle.num_threads(), kind="oracle",
                sample=f"{n} run(s) of a {rows}-token chunk of one sequence in {el:.1f} s (fp64 oracle)")


def bench_compressed(torch, nd, steps, warmup, pk, dist=None, cpu_budget=None, block=4):
    from workloads import compressed
    w = compressed()
    w["block"] = block
    B, T, H, d = w["q"].shape
    q, k, v = dev_bf16(torch, w["q_bits"]), dev_bf16(torch, w["k_bits"]), dev_bf16(torch, w["v_bits"])
    nb = T // block
    pkk = torch.empty((B, nb, H, d), dtype=torch.bfloat16, device="cuda")
    pvv = torch.empty_like(pkk)
    out = torch.empty_like(q)
    nbytes = nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, H, H, d, w["rope_theta"], block)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")

    def step(i):   # one call: pooling fused with K's rotation, then the attention
        nd.nd_swa_sink_prefill(q, k, v, None, None, w["window"], rope_theta=w["rope_theta"], block=block, out=out,
                               workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    nd.nd_kv_compress_pool(k, v, block, w["rope_theta"], pooled_k=pkk, pooled_v=pvv)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    nd.nd_rope_apply(q, qr, w["rope_theta"])
    nd.nd_rope_apply(k, kr, w["rope_theta"])
    ws0 = torch.empty(max(nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, H, H, d, 0.0, block), 16),
                      dtype=torch.uint8, device="cuda")

    def attn(i):
        nd.nd_swa_sink_prefill(qr, kr, v, None, None, w["window"], rope_theta=0.0, pooled_k=pkk, pooled_v=pvv,
                               block=block, out=out, workspace=ws0)

    ms_attn = time_graph(torch, attn, steps, warmup, dist)
    tiles = nd.nd_swa_sink_prefill_tiles(ws0, B, T, H, H, d, 0.0, block)
    pairs = visible_pairs_compressed(T, w["window"], block) * B * H
    flops = 4.0 * d * pairs
    tile_flops = 4.0 * 128 * 64 * d * tiles
    t, ta = ms / steps, ms_attn / steps
    oracle_row = None
    if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
        try:
            oracle_row = oracle_prefill_sample("compressed", w, 2, 2, cpu_budget)
        except Exception as ex:  # the product path never depends on it
            oracle_row = {"tok_s": None, "sample": f"unavailable: {ex}"}
    return dict(config=f"compressed prefill B{B} T{T} H{H} d{d} W256 b{block} RoPE, one call (pooling fused with "
                       f"K's rotation, then attention)",
                oracle=oracle_row, ms_per_step=t, tok_s=B * T / (t * 1e-3), step_tflops=flops / (t * 1e-3) / 1e12,
                visible_pairs=pairs, attn_ms=ta,
                attn_algorithmic=roofline("tensor", flops, ta, pk["bf16"], "TFLOP/s",
                                          "prefill_tc_kernel (visible pairs)", pk["src"]),
                tiles=tiles, tile_flops=tile_flops, tile_overhead=tile_flops / flops,
                roofline=roofline("tensor", tile_flops, ta, pk["bf16"], "TFLOP/s",
                                  "prefill_tc_kernel (tiles its plan performed)", pk["src"],
                                  load_traffic(f"prefill_tc@compressed_b{block}")),
                launches=4 * steps)


def visible_pairs_pinned(T, W, b, P):
    """Visible (query, column) pairs of one (sequence, head) of the pinned
    compressed prefill: pinned keys, exact window keys past the pins, and
    the visible pooled blocks of the positions after the pins."""
    t = np.arange(T)
    pinned = np.minimum(t + 1, P)
    lo = np.maximum(t - W + 1, P)
    exact = np.clip(t - lo + 1, 0, None)
    pooled = np.clip((t - W + 1 - P) // b, 0, (T - P) // b)
    return int((pinned + exact + pooled).sum())


def bench_compressed_pinned(torch, nd, steps, warmup, pk, dist=None, block=4, n_pinned=512):
    """The compressed prefill with a pinned prefix (the first n_pinned
    positions exact and visible at any distance, blocks pooled after them):
    one nd_compressed_prefill call (fused pooling + rotation, attention)."""
    from workloads import compressed
    w = compressed()
    B, T, H, d = w["q"].shape
    q, k, v = dev_bf16(torch, w["q_bits"]), dev_bf16(torch, w["k_bits"]), dev_bf16(torch, w["v_bits"])
    out = torch.empty_like(q)
    ws = torch.empty(nd.nd_compressed_prefill_workspace_size(B, T, H, H, d, w["rope_theta"], block), dtype=torch.uint8,
                     device="cuda")

    def step(i):
        nd.nd_compressed_prefill(q, k, v, w["window"], block, n_pinned=n_pinned, rope_theta=w["rope_theta"], out=out,
                                 workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    tiles = nd.nd_swa_sink_prefill_tiles(ws, B, T, H, H, d, w["rope_theta"], block)
    pairs = visible_pairs_pinned(T, w["window"], block, n_pinned) * B * H
    flops = 4.0 * d * pairs
    tile_flops = 4.0 * 128 * 64 * d * tiles
    return dict(config=f"compressed prefill with a {n_pinned}-token pinned prefix, B{B} T{T} H{H} d{d} W256 b{block} "
                       f"RoPE, one call", ms_per_step=t, tok_s=B * T / (t * 1e-3), visible_pairs=pairs, tiles=tiles,
                tile_overhead=tile_flops / flops,
                algorithmic=roofline("tensor", flops, t, pk["bf16"], "TFLOP/s", "whole call (visible pairs)", pk["src"]),
                roofline=roofline("tensor", tile_flops, t, pk["bf16"], "TFLOP/s",
                                  "whole call (tiles the attention kernel's plan performed)", pk["src"]),
                launches=4 * steps)


def bench_tiny_fp32(torch, nd, steps, warmup, pk, dist=None, cpu_budget=None):
    """fp32 tiny prefill (B1 T512 Hq4 Hkv1 d64, W256; literal segments and the
    single-segment variant) on CUDA cores: FLOP/s against the fp32 FFMA peak."""
    import oracle
    from workloads import tiny_prefill
    res = {}
    for name, single in (("literal", False), ("single_segment", True)):
        w = tiny_prefill(single_segment=single)
        q, k, v = (torch.from_numpy(w[x]).cuda() for x in ("q", "k", "v"))
        seg, sink = torch.from_numpy(w["seg_ids"]).cuda(), torch.from_numpy(w["sink"]).cuda()
        out = torch.empty_like(q)
        B_, T_, Hq_, d_ = q.shape
        nbytes = nd.nd_swa_sink_prefill_workspace_size(nd.ND_F32, B_, T_, Hq_, k.shape[2], d_, 0.0, 0)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")

        def step(i):
            nd.nd_swa_sink_prefill(q, k, v, seg, sink, w["window"], out=out, workspace=ws)

        ms = time_graph(torch, step, steps, warmup, dist)
        t = ms / steps
        pairs = int(visible_pairs_packed(w["seg_ids"], w["sink"], w["window"]).sum())
        flops = 4.0 * 64 * pairs * 4
        orow = None
        if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
            n, t0 = 0, time.perf_counter()
            while True:
                oracle.swa_sink_prefill(w["q"], w["k"], w["v"], w["seg_ids"], w["sink"], w["window"])
                n += 1
                if time.perf_counter() - t0 >= cpu_budget:
                    break
            el = time.perf_counter() - t0
            orow = dict(tok_s=512 * n / el, cores=oracle.num_threads(), kind="oracle",
                        sample=f"{n} full runs in {el:.1f} s")
        res[name] = dict(ms_per_call=t, visible_pairs=pairs, tok_s=512 / (t * 1e-3), oracle=orow,
                         roofline=roofline("alu", flops, t, alu_fp32_peak_tflops(), "TFLOP/s",
                                           "prefill_simt_kernel (fp32 FFMA)", "derived: 152 SMs x 128 FP32 lanes x "
                                           "2 flops x 2.07 GHz", load_traffic(f"prefill_simt@tiny_{name}")))
    return dict(config="tiny prefill B1 T512 Hq4 Hkv1 d64 fp32, 48-token sink prefix, W256", **res)


# ----------------------------------------------------------------------------
# pooling, append, handoff
# ----------------------------------------------------------------------------

def bench_pool(torch, nd, steps, warmup, pk, dist=None, block=4, cpu_budget=None):
    """Block pooling with midpoint rotation alone (the compressed workload's
    K and V), rotating replicas of the inputs."""
    import oracle
    from workloads import compressed
    w = compressed()
    B, T, H, d = w["k"].shape
    nb = T // block
    per = 2 * B * T * H * d * 2 + 2 * B * nb * H * d * 2
    replicas = max(1, math.ceil(4 * L2_BYTES / per))
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    reps = []
    for _ in range(replicas):
        k = torch.randn((B, T, H, d), generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn((B, T, H, d), generator=g, device="cuda").to(torch.bfloat16)
        reps.append((k, v, torch.empty((B, nb, H, d), dtype=torch.bfloat16, device="cuda"),
                     torch.empty((B, nb, H, d), dtype=torch.bfloat16, device="cuda")))

    def step(i):
        k, v, pkk, pvv = reps[i % replicas]
        nd.nd_kv_compress_pool(k, v, block, w["rope_theta"], pooled_k=pkk, pooled_v=pvv)

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    orow = None
    if int(os.environ.get("RANK", "0")) == 0 and cpu_budget is not None:
        n, t0 = 0, time.perf_counter()
        kk = w["k"][:1].astype(np.float64)
        while True:
            oracle.compress(kk, kk, kk, block, w["rope_theta"])
            n += 1
            if time.perf_counter() - t0 >= cpu_budget:
                break
        el = time.perf_counter() - t0
        orow = dict(gbs=per / B * n / el / 1e9, cores=1, kind="oracle",
                    sample=f"{n} runs of one sequence's pooling (and rotation of its keys) in {el:.1f} s, "
                           "bytes of one sequence")
    return dict(config=f"block pooling + midpoint rotation, B{B} T{T} H{H} d{d} b{block} (K and V)",
                ms_per_launch=t, bytes_per_launch=per, replicas=replicas, oracle=orow,
                roofline=roofline("hbm", per, t, pk["hbm"], "GB/s", "pool_vec_kernel", pk["src"],
                                  load_traffic(f"pool@compressed_b{block}")))


def bench_pool_rope(torch, nd, steps, warmup, pk, dist=None, block=4):
    """The compressed prefill's fused pass over K and V alone
    (nd_kv_compress_pool_rope: angle table, then K rotated at every position
    and the pooled blocks), rotating replicas of the inputs."""
    from workloads import compressed
    w = compressed()
    B, T, H, d = w["k"].shape
    nb = T // block
    per = 2 * B * T * H * d * 2 + B * T * H * d * 2 + 2 * B * nb * H * d * 2
    replicas = max(1, math.ceil(4 * L2_BYTES / per))
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    reps = []
    for _ in range(replicas):
        k = torch.randn((B, T, H, d), generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn((B, T, H, d), generator=g, device="cuda").to(torch.bfloat16)
        reps.append((k, v, torch.empty_like(k), torch.empty((B, nb, H, d), dtype=torch.bfloat16, device="cuda"),
                     torch.empty((B, nb, H, d), dtype=torch.bfloat16, device="cuda")))
    ws = torch.empty(nd.nd_kv_compress_pool_rope_workspace_size(T, d, w["rope_theta"]), dtype=torch.uint8,
                     device="cuda")

    def step(i):
        k, v, kr, pkk, pvv = reps[i % replicas]
        nd.nd_kv_compress_pool_rope(k, v, block, w["rope_theta"], k_rot=kr, pooled_k=pkk, pooled_v=pvv, workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    return dict(config=f"pooling fused with K's rotation, B{B} T{T} H{H} d{d} b{block}: read K and V once, write "
                       f"rotated K and the pooled blocks (+ the 0.5 MB angle table)",
                ms_per_step=t, bytes_per_launch=per, replicas=replicas,
                roofline=roofline("hbm", per, t, pk["hbm"], "GB/s", "rope_table_kernel + pool_rope_bulk_kernel", pk["src"],
                                  load_traffic(f"pool_rope@compressed_b{block}")))


def bench_append(torch, nd, steps, warmup, pk, dist=None, B=512, Hkv=8, d=128, S=1024, W=256):
    """Standalone quantise-and-append of one token per sequence into the
    large-batch cache (new tokens rotate through buffers larger than L2)."""
    cache = nd.KVCache.empty(B, Hkv, d, S, W)
    cache.sink_len.fill_(S)
    cache.ring_len.fill_(W)
    cache.seq_len.fill_(S + W)
    per = B * Hkv * (2 * d * 2 + 2 * d + 2 * (d // 32) * 4)
    n_tok = max(1, math.ceil(4 * L2_BYTES / (B * Hkv * d * 2 * 2)))
    toks = [(torch.randn((B, Hkv, d), device="cuda").to(torch.bfloat16),
             torch.randn((B, Hkv, d), device="cuda").to(torch.bfloat16)) for _ in range(n_tok)]

    def step(i):
        kn, vn = toks[i % n_tok]
        nd.nd_kv_append_quant(cache, kn, vn, False)

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    return dict(config=f"quantise-and-append of one bf16 token per sequence, B{B} Hkv{Hkv} d{d} "
                       f"into {S} sinks + {W} ring", ms_per_launch=t, bytes_per_launch=per,
                roofline=roofline("hbm", per, t, pk["hbm"], "GB/s", "kv_append_quant_kernel", pk["src"]))


def fill_kept_tokens(seg, sink, S, W):
    """Tokens the handoff writes per (batch row, segment) under the append
    rule for the packed workload's layout (segments are runs that open with
    their sink prefix)."""
    kept = 0
    entries = 0
    for b in range(seg.shape[0]):
        for s in np.unique(seg[b]):
            if s <= 0:
                continue
            idx = np.nonzero(seg[b] == s)[0]
            sk = sink[b, idx] != 0
            f = int(np.argmin(sk)) if not sk.all() else len(idx)   # first ring token
            n_ring = int((~sk).sum())
            kept += min(f, S) + min(n_ring, W)
            entries += 1
    return kept, entries


def bench_fill(torch, nd, steps, warmup, pk, dist=None, S=512, W=256):
    """Prefill -> cache handoff of the packed workload (every segment of every
    row), rotating replicas of the prefill's K/V."""
    from workloads import packed_prefill
    w = packed_prefill()
    B, T, Hkv, d = w["k"].shape
    seg, sink = w["seg_ids"], w["sink"]
    kept, n = fill_kept_tokens(seg, sink, S, W)
    src_row = torch.tensor([b for b in range(B) for s in np.unique(seg[b]) if s > 0], dtype=torch.int32, device="cuda")
    src_seg = torch.tensor([int(s) for b in range(B) for s in np.unique(seg[b]) if s > 0], dtype=torch.int32,
                           device="cuda")
    per = kept * Hkv * (2 * d * 2 + 2 * d + 2 * (d // 32) * 4) + B * T * 5
    replicas = 4
    k0, v0 = dev_bf16(torch, w["k_bits"]), dev_bf16(torch, w["v_bits"])
    kvs = [(k0, v0)] + [(k0.roll(r, 1).contiguous(), v0.roll(r, 1).contiguous()) for r in range(1, replicas)]
    caches = [nd.KVCache.empty(n, Hkv, d, S, W) for _ in range(replicas)]
    seg_d, sink_d = torch.from_numpy(seg).cuda(), torch.from_numpy(sink).cuda()
    ws = torch.empty(nd.nd_kv_cache_from_prefill_workspace_size(n, S, W), dtype=torch.uint8, device="cuda")

    def step(i):
        k, v = kvs[i % replicas]
        nd.nd_kv_cache_from_prefill(caches[i % replicas], k, v, src_row, seg_d, sink_d, src_seg, workspace=ws)

    ms = time_graph(torch, step, steps, warmup, dist)
    t = ms / steps
    return dict(config=f"prefill->cache handoff of the packed workload (B{B} T{T} Hkv{Hkv} d{d}, {n} segments) "
                       f"into {S} sink + {W} ring slots per segment", ms_per_launch=t, kept_tokens=kept,
                bytes_per_launch=per, replicas=replicas,
                roofline=roofline("hbm", per, t, pk["hbm"], "GB/s", "kv_fill_plan_kernel + kv_fill_kernel",
                                  pk["src"], load_traffic("cache_handoff@packed")))


# ----------------------------------------------------------------------------
# CPU baseline (the oracle on the host cores)
# ----------------------------------------------------------------------------

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


def oracle_decode_sample(B, Hq, Hkv, d, S, W, seed, budget_s, of_batch=None):
    """Times the oracle's decode on the host: B sequences of the workload (a
    sample of its of_batch), one full decode of all B per iteration, repeated
    until budget_s elapses; GB/s of the sample's cache bytes."""
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
    threads = min(oracle.num_threads(), B)   # the oracle takes whole sequences per thread
    what = f"{B} of the {of_batch} sequences" if of_batch else f"all {B} sequences"
    return dict(value=(cache_b + qo_b) * n / el / 1e9, unit="GB/s", cores=threads, kind="oracle",
                sample=f"{n} decode(s) of {what} of the Hq{Hq} Hkv{Hkv} d{d} S{S}+W{W} workload in {el:.1f} s "
                       f"(fp64 dense oracle, OpenMP over sequences); GB/s of those sequences' cache bytes",
                seconds=el / n)


# ----------------------------------------------------------------------------

HEAD = dict(B=512, Hq=32, Hkv=8, d=128, S=1024, W=256)
ORACLE_SAMPLE = 32   # sequences of the headline workload the oracle decodes per step
ALL_ROWS = ("step_b64", "sweep", "wsweep", "packed", "compressed", "compressed_b8", "compressed_pinned", "tiny",
            "pool", "pool_rope", "append", "fill", "cdecode", "chunk")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nd", choices=["nd", "reference"])
    ap.add_argument("--rows", default="all", help="comma list of rows (" + ",".join(ALL_ROWS) + "), all or none")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--sweep-batches", default="32,64,128,256",
                    help="batch sizes of the decode sweep besides the headline's 512")
    ap.add_argument("--packed-batch", type=int, default=8,
                    help="sequences in the packed-prefill row (8 = the measured configuration; smaller for profiling)")
    ap.add_argument("--head-batch", type=int, default=HEAD["B"],
                    help="sequences of the headline decode step (512 = the measured configuration; smaller for "
                         "profiling)")
    ap.add_argument("--cdecode-batch", type=int, default=128,
                    help="sequences of the compressed-decode row (128 = the measured configuration)")
    ap.add_argument("--chunk-batch", type=int, default=8,
                    help="sequences of the chunked-prefill row (8 = the measured configuration)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    h = dict(HEAD, B=args.head_batch)
    workload = (f"decode step B{h['B']} Hq{h['Hq']} Hkv{h['Hkv']} d{h['d']}, {h['S']} sink slots + {h['W']}-slot ring "
                f"(full, random offset), int8 g32 K/V, quantise-and-append of one bf16 token per sequence")

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        per_step = []
        for i in range(warmup + steps):
            r = oracle_decode_sample(ORACLE_SAMPLE, h["Hq"], h["Hkv"], h["d"], h["S"], h["W"], 1234 + 4,
                                     budget_s=0.0, of_batch=h["B"])
            if i >= warmup:
                per_step.append(r["seconds"])
        ms = 1e3 * sum(per_step) / len(per_step)
        cache_b, qo_b, _ = decode_bytes(ORACLE_SAMPLE, h["Hq"], h["Hkv"], h["d"], h["S"], h["W"])
        val = (cache_b + qo_b) / (ms * 1e-3) / 1e9
        line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus, "steps": steps,
                "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": {"workload": workload, "l2": "host run"},
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": f"each step is one oracle decode of {ORACLE_SAMPLE} of the workload's "
                                           f"{h['B']} sequences (fp64, OpenMP over sequences)"},
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
    want = set(ALL_ROWS) if args.rows == "all" else (set() if args.rows == "none" else set(args.rows.split(",")))
    budget = None if rank != 0 else min(3.0, args.cpu_budget)

    with ClockSampler(dev_index) as clk:
        head = bench_decode(torch, nd, h["B"], h["Hq"], h["Hkv"], h["d"], h["S"], h["W"], steps, warmup,
                            seed=rank_seed(1234 + 4, rank), pk=pk, dist=dist, traffic_key=f"decode@decode_b{h['B']}")
    clocks = clk.summary()
    e2e = e2e_decode(torch, nd, head.pop("_state"), h["B"], h["Hq"], h["Hkv"], h["d"], h["S"], h["W"],
                     min(steps, 50), warmup)
    torch.cuda.empty_cache()

    rows = {}
    row_steps = max(10, steps // 10)
    if "step_b64" in want:
        r = bench_decode(torch, nd, 64, 8, 2, 64, 64, 256, steps, warmup, seed=rank_seed(1234 + 1, rank), pk=pk,
                         dist=dist, traffic_key="decode_step@decode_b64")
        r["e2e"] = e2e_decode(torch, nd, r.pop("_state"), 64, 8, 2, 64, 64, 256, min(steps, 200), warmup)
        if budget:
            r["oracle"] = oracle_decode_sample(64, 8, 2, 64, 64, 256, 1234 + 1, budget)
        rows["decode_step_b64"] = r
        torch.cuda.empty_cache()
    if "sweep" in want:
        sweep = {}
        for Bs in [int(x) for x in args.sweep_batches.split(",") if x]:
            r = bench_decode(torch, nd, Bs, 32, 8, 128, 1024, 256, max(20, steps // 4), warmup,
                             seed=rank_seed(1234 + 4, rank), pk=pk, dist=dist, traffic_key=f"decode@decode_b{Bs}")
            r.pop("_state")
            sweep[f"B{Bs}"] = {k: r[k] for k in ("ms_per_step", "gbs", "frac", "decode_kernel_gbs",
                                                 "decode_kernel_frac", "replicas", "roofline")}
            torch.cuda.empty_cache()
        sweep["B512"] = {k: head[k] for k in ("ms_per_step", "gbs", "frac", "decode_kernel_gbs",
                                              "decode_kernel_frac", "replicas", "roofline")}
        rows["decode_sweep"] = dict(config="decode step, Hq32 Hkv8 d128, 1024 sinks + 256 ring; B512 is the headline",
                                    oracle="as cpu_baseline (same workload per sequence)", **sweep)
    if "wsweep" in want:
        rows["window_sweep"] = bench_window_sweep(torch, nd, max(20, steps // 4), warmup, pk, dist)
    if "packed" in want:
        rows["packed_prefill"] = bench_packed_prefill(torch, nd, row_steps, warmup, pk, dist, batch=args.packed_batch,
                                                      cpu_budget=budget)
        torch.cuda.empty_cache()
    if "compressed" in want:
        rows["compressed_prefill"] = bench_compressed(torch, nd, row_steps, warmup, pk, dist, cpu_budget=budget)
        torch.cuda.empty_cache()
    if "compressed_b8" in want:
        rows["compressed_prefill_b8"] = bench_compressed(torch, nd, row_steps, warmup, pk, dist, cpu_budget=budget,
                                                         block=8)
        torch.cuda.empty_cache()
    if "compressed_pinned" in want:
        rows["compressed_prefill_pinned"] = bench_compressed_pinned(torch, nd, row_steps, warmup, pk, dist)
        torch.cuda.empty_cache()
    if "tiny" in want:
        rows["tiny_prefill_fp32"] = bench_tiny_fp32(torch, nd, row_steps, warmup, pk, dist,
                                                    cpu_budget=None if budget is None else 1.0)
    if "pool" in want:
        rows["pool"] = bench_pool(torch, nd, row_steps, warmup, pk, dist, cpu_budget=None if budget is None else 1.0)
        torch.cuda.empty_cache()
    if "pool_rope" in want:
        rows["pool_rope"] = bench_pool_rope(torch, nd, row_steps, warmup, pk, dist)
        torch.cuda.empty_cache()
    if "append" in want:
        rows["append"] = bench_append(torch, nd, max(20, steps // 4), warmup, pk, dist)
        torch.cuda.empty_cache()
    if "fill" in want:
        rows["cache_handoff"] = bench_fill(torch, nd, row_steps, warmup, pk, dist)
        torch.cuda.empty_cache()
    if "chunk" in want:
        rows["chunk_prefill"] = bench_chunk(torch, nd, row_steps, warmup, pk, dist, B=args.chunk_batch,
                                            cpu_budget=budget)
        torch.cuda.empty_cache()
    if "cdecode" in want:
        rows["compressed_decode"] = bench_compressed_decode(torch, nd, max(20, steps // 4), warmup, pk, dist,
                                                            B=args.cdecode_batch)
        torch.cuda.empty_cache()

    value = job_throughput(head["bytes_per_step"], steps, world, head["ms_per_step"] * steps)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 KV / bf16 q,out / fp32 accum", "data": "synthetic",
        "config": {"workload": workload,
                   "l2": f"inputs larger than L2 ({head['bytes_per_step'] / 1e9:.2f} GB per step, "
                         f"{head['replicas']} cache replica(s))",
                   "timing": "CUDA graph of K steps, CUDA events"},
        "step": {"gbs": head["gbs"], "frac": head["frac"], "launches_per_step": head["launches"] // steps},
        "roofline": head["roofline"],
        "gpu_launches": head["launches"],
        "clocks": clocks,
        "e2e": e2e,
        "rows": rows,
    }
    if rank == 0:
        try:
            cb = oracle_decode_sample(min(ORACLE_SAMPLE, h["B"]), h["Hq"], h["Hkv"], h["d"], h["S"], h["W"], 1234 + 4,
                                      args.cpu_budget, of_batch=h["B"])
            cb.pop("seconds", None)
            line["cpu_baseline"] = cb
        except Exception as ex:  # the product path never depends on it
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 0, "kind": "oracle",
                                    "sample": f"unavailable: {ex}"}
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
