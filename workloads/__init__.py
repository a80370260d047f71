"""Seeded synthetic inputs shared by the tests and the benchmark.

This module draws random numbers and lays out segments; it holds none of the
method's arithmetic (no masking, softmax, quantisation, pooling or rotation).
Every generator is a numpy Philox (counter-based) stream keyed by an integer
seed, so the same seed gives the same bits on x86 and on Arm.  bf16 tensors are
returned as their uint16 bit patterns (round-to-nearest-even from fp32) next to
the exact fp32 widening of those bits, so the CUDA path and the oracle read the
same values.

Workloads (sizes and distributions of the five measured configurations):
  tiny_prefill      B1 T512 Hq4 Hkv1 d64 fp32, seg 1 = 48-token sink prefix,
                    seg 2 = the rest (or one segment with the same sink), W256
  decode_cache      K/V tokens N(0,1) bf16 for S sink + W ring slots per
                    sequence, random ring offset, bf16 query N(0,1)
  packed_prefill    B8 T4096 Hq32 Hkv8 d128 bf16 N(0,1); each row packs 3-6
                    segments with uniform cut points (every segment >= 513
                    tokens), each opening with a sink prefix of 64-512 tokens
  compressed        B4 T4096 H16 d64 bf16 N(0,1), pre-rotation q/k/v
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 1234


def philox(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def to_bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit pattern -> fp32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape):
    """N(0,1) rounded to bf16: (bits uint16, exact fp32 values)."""
    bits = to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    return bits, bf16_bits_to_f32(bits)


def packed_segments(rng: np.random.Generator, B: int, T: int, n_min: int = 3,
                    n_max: int = 6, min_len: int = 513, sink_min: int = 64,
                    sink_max: int = 512):
    """Segment ids (1..n, consecutive runs tiling T) and a sink flag per
    position: every segment opens with a sink prefix of U{sink_min..sink_max}
    tokens (capped at the segment length).  Cut points are uniform; a draw is
    rejected until every segment has at least min_len tokens."""
    seg = np.zeros((B, T), np.int32)
    sink = np.zeros((B, T), np.uint8)
    for b in range(B):
        n = int(rng.integers(n_min, n_max + 1))
        while True:
            cuts = np.sort(rng.choice(np.arange(1, T), size=n - 1, replace=False))
            bounds = np.concatenate(([0], cuts, [T]))
            if np.all(np.diff(bounds) >= min_len):
                break
        for i in range(n):
            s, e = int(bounds[i]), int(bounds[i + 1])
            seg[b, s:e] = i + 1
            ns = min(int(rng.integers(sink_min, sink_max + 1)), e - s)
            sink[b, s:s + ns] = 1
    return seg, sink


def tiny_prefill(single_segment: bool = False, seed: int = BASE_SEED + 0, T: int = 512,
                 Hq: int = 4, Hkv: int = 1, d: int = 64, n_sink: int = 48):
    """fp32 q/k/v N(0,1); seg 1 = [0, n_sink) marked sink, seg 2 = the rest
    (single_segment: one segment, same sink prefix)."""
    rng = philox(seed)
    q = rng.standard_normal((1, T, Hq, d), dtype=np.float32)
    k = rng.standard_normal((1, T, Hkv, d), dtype=np.float32)
    v = rng.standard_normal((1, T, Hkv, d), dtype=np.float32)
    seg = np.full((1, T), 1 if single_segment else 2, np.int32)
    seg[0, :n_sink] = 1
    sink = np.zeros((1, T), np.uint8)
    sink[0, :n_sink] = 1
    return dict(q=q, k=k, v=v, seg_ids=seg, sink=sink, window=256)


def decode_cache(B: int, Hq: int, Hkv: int, d: int, sink_cap: int, ring_cap: int,
                 seed: int, full: bool = True):
    """Raw (pre-quantisation) K/V token values for every cache slot, a bf16
    query per sequence, and cache metadata: every sink slot filled, the ring
    full (or a random fill when full=False) with a random physical offset."""
    rng = philox(seed)
    ns = sink_cap + ring_cap
    k_bits, k = normal_bf16(rng, (B, Hkv, ns, d))
    v_bits, v = normal_bf16(rng, (B, Hkv, ns, d))
    q_bits, q = normal_bf16(rng, (B, Hq, d))
    ring_start = rng.integers(0, ring_cap, size=B).astype(np.int32)
    if full:
        ring_len = np.full(B, ring_cap, np.int32)
    else:
        ring_len = rng.integers(1, ring_cap + 1, size=B).astype(np.int32)
    sink_len = np.full(B, sink_cap, np.int32)
    # Tokens seen: the sinks, then ring appends; a ring that wrapped r times
    # past its start has seen ring_len + ring_start appends.
    seq_len = (sink_len + ring_len + np.where(ring_len == ring_cap, ring_start, 0)).astype(np.int32)
    if not full:
        ring_start = np.zeros(B, np.int32)
    return dict(k_bits=k_bits, k=k, v_bits=v_bits, v=v, q_bits=q_bits, q=q,
                sink_len=sink_len, ring_start=ring_start, ring_len=ring_len,
                seq_len=seq_len)


def decode_b64(seed: int = BASE_SEED + 1):
    """Decode step: B64 Hq8 Hkv2 d64, 64 sink slots + full 256-slot ring."""
    return decode_cache(64, 8, 2, 64, 64, 256, seed)


def decode_sweep(B: int, seed: int = BASE_SEED + 4):
    """Large-batch decode: Hq32 Hkv8 d128, 1024 sink slots + full 256 ring."""
    return decode_cache(B, 32, 8, 128, 1024, 256, seed)


def random_codes(rng: np.random.Generator, B: int, Hkv: int, ns: int, d: int):
    """Directly drawn cache contents for sizes where quantising N(0,1) tokens
    on the host is too slow: codes uniform in [-127, 127], scales the absmax/127
    of N(0,1) groups would give (about 2.2/127..3.3/127)."""
    kc = rng.integers(-127, 128, size=(B, Hkv, ns, d), dtype=np.int8)
    vc = rng.integers(-127, 128, size=(B, Hkv, ns, d), dtype=np.int8)
    ks = rng.uniform(2.2 / 127, 3.3 / 127, size=(B, Hkv, ns, d // 32)).astype(np.float32)
    vs = rng.uniform(2.2 / 127, 3.3 / 127, size=(B, Hkv, ns, d // 32)).astype(np.float32)
    return kc, ks, vc, vs


def packed_prefill(seed: int = BASE_SEED + 2, B: int = 8, T: int = 4096, Hq: int = 32,
                   Hkv: int = 8, d: int = 128, n_min: int = 3, n_max: int = 6,
                   min_len: int = 513, sink_min: int = 64, sink_max: int = 512):
    """Packed-segment prefill inputs (bf16 bits + fp32 values)."""
    rng = philox(seed)
    seg, sink = packed_segments(rng, B, T, n_min, n_max, min_len, sink_min, sink_max)
    q_bits, q = normal_bf16(rng, (B, T, Hq, d))
    k_bits, k = normal_bf16(rng, (B, T, Hkv, d))
    v_bits, v = normal_bf16(rng, (B, T, Hkv, d))
    return dict(q_bits=q_bits, q=q, k_bits=k_bits, k=k, v_bits=v_bits, v=v,
                seg_ids=seg, sink=sink, window=256, rope_theta=10000.0)


def compressed(seed: int = BASE_SEED + 3, B: int = 4, T: int = 4096, H: int = 16,
               d: int = 64):
    """Compressed-attention inputs, pre-rotation (bf16 bits + fp32 values)."""
    rng = philox(seed)
    q_bits, q = normal_bf16(rng, (B, T, H, d))
    k_bits, k = normal_bf16(rng, (B, T, H, d))
    v_bits, v = normal_bf16(rng, (B, T, H, d))
    return dict(q_bits=q_bits, q=q, k_bits=k_bits, k=k, v_bits=v_bits, v=v,
                window=256, block=4, rope_theta=10000.0)
