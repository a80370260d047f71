"""GPU parity: the prefill -> cache handoff (nd_kv_cache_from_prefill).

A cache row filled from segment s of batch row b must hold exactly what the
oracle's append (kv_append) leaves after appending that segment's tokens one
at a time, in position order, with to_sink = sink[b][t], to an empty row:
codes, scales and metadata bit-exact ("KV Sinks for Tools": the pinned prefix
stays, the ring keeps the newest positions).  A decode step after the handoff
then matches the oracle's decode on the replayed cache."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev, dev_bf16, host, need_gpu, no_device_errors
from workloads import bf16_bits_to_f32, normal_bf16, packed_prefill, packed_segments, philox, to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    no_device_errors()


def nd():
    import sliding_window_kv_swa_gb300 as m
    return m


def replay(k, v, seg, sink, entries, Hkv, d, S, W):
    """Oracle cache (one row per entry) after appending each entry's segment
    tokens in order; returns (cache, rejected sink tokens per entry)."""
    n = len(entries)
    ref = oracle.Cache(n, Hkv, d, S, W)
    rejected = []
    for e, (b, s) in enumerate(entries):
        one = oracle.Cache(1, Hkv, d, S, W)
        ts = np.nonzero(seg[b] == s)[0] if seg is not None else np.arange(k.shape[1])
        rej = 0
        for t in ts:
            rej += oracle.kv_append(one, k[b, t][None], v[b, t][None], bool(sink is not None and sink[b, t]))
        rejected.append(rej)
        for f in ("k_codes", "v_codes", "k_scale", "v_scale"):
            getattr(ref, f)[e] = getattr(one, f)[0]
        for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
            getattr(ref, f)[e] = getattr(one, f)[0]
    return ref, rejected


def compare_filled(cache, ref, rows):
    """Metadata of every filled row, and the codes and scales of its occupied
    slots (the replay starts from zeros; other slots are not visible)."""
    S = ref.sink_cap
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        np.testing.assert_array_equal(host(getattr(cache, f))[rows], getattr(ref, f)[rows], err_msg=f)
    got = {f: host(getattr(cache, f)) for f in ("k_codes", "v_codes", "k_scale", "v_scale")}
    for e in rows:
        occ = list(range(int(ref.sink_len[e]))) + [S + r for r in range(int(ref.ring_len[e]))]
        for f in got:
            np.testing.assert_array_equal(got[f][e][:, occ], getattr(ref, f)[e][:, occ], err_msg=f"{f} row {e}")


@pytest.mark.parametrize("d,Hkv", [(64, 2), (128, 3), (32, 1), (64, 3), (256, 2)])
def test_fill_matches_oracle_replay(d, Hkv):
    rng = philox(3000 + d)
    B, T, S, W = 2, 700, 160, 48
    kb, kf = normal_bf16(rng, (B, T, Hkv, d))
    vb, vf = normal_bf16(rng, (B, T, Hkv, d))
    seg, sink = packed_segments(rng, B, T, 2, 3, T // 4, 3, T // 8)
    entries = [(b, int(s)) for b in range(B) for s in np.unique(seg[b]) if s > 0]
    # plus a row left untouched (src_row = -1)
    src_row = np.array([b for b, _ in entries] + [-1], np.int32)
    src_seg = np.array([s for _, s in entries] + [1], np.int32)
    n = len(src_row)
    cache = nd().KVCache.empty(n, Hkv, d, S, W)
    cache.k_codes.fill_(7)
    cache.sink_len[n - 1] = 5
    before = host(cache.k_codes[n - 1]).copy()
    nd().nd_kv_cache_from_prefill(cache, dev_bf16(kb), dev_bf16(vb), dev(src_row), dev(seg), dev(sink),
                                  dev(src_seg))
    ref, rejected = replay(kf, vf, seg, sink, entries, Hkv, d, S, W)
    assert sum(rejected) == 0
    compare_filled(cache, ref, list(range(n - 1)))
    np.testing.assert_array_equal(host(cache.k_codes[n - 1]), before)
    assert int(host(cache.sink_len)[n - 1]) == 5


@pytest.mark.parametrize("T", [4099, 8200])
def test_fill_rows_longer_than_one_planning_pass(T):
    """Batch rows longer than the planner's single pass of 4096 positions
    (both walks then loop), with and without a whole number of 4-position
    quads per row."""
    rng = philox(3050 + T)
    B, Hkv, d, S, W = 1, 1, 32, 64, 96
    kb, kf = normal_bf16(rng, (B, T, Hkv, d))
    vb, vf = normal_bf16(rng, (B, T, Hkv, d))
    seg = np.ones((B, T), np.int32)
    seg[0, T // 3:] = 2
    seg[0, T - 50:] = 0                                   # trailing padding
    sink = np.zeros((B, T), np.uint8)
    sink[0, :40] = 1                                      # segment 1: 40 sinks
    sink[0, T // 3:T // 3 + 70] = 1                       # segment 2: 70 sinks > S (rejected past 64)
    entries = [(0, 1), (0, 2)]
    src_row = np.array([b for b, _ in entries], np.int32)
    src_seg = np.array([s for _, s in entries], np.int32)
    cache = nd().KVCache.empty(len(entries), Hkv, d, S, W)
    nd().nd_kv_cache_from_prefill(cache, dev_bf16(kb), dev_bf16(vb), dev(src_row), dev(seg), dev(sink),
                                  dev(src_seg))
    assert nd().nd_device_errors(clear=True) == 2          # segment 2's rejected sinks (metadata flag)
    ref, rejected = replay(kf, vf, seg, sink, entries, Hkv, d, S, W)
    assert rejected == [0, 6]
    compare_filled(cache, ref, list(range(len(entries))))


def test_fill_codes_at_and_beside_half_integer_quotients():
    """The handoff's quantiser on groups whose quotients x / scale sit exactly
    on half-integers (ties to even) and one or two bf16 steps either side,
    at several scales, plus a group whose scale is subnormal (the quotient
    path and its clamp) and an all-zero group: codes and scales bit for bit
    against the oracle's codec, through a whole-row handoff."""
    groups = []
    for k in (-20, -3, 0, 5, 17):
        sc = 2.0 ** k
        for n in range(-127, 127, 3):
            base = (n + 0.5) * sc
            vals = [base]
            b = to_bf16_bits(np.array([base], np.float32)).astype(np.int32)[0]
            for dlt in (-2, -1, 1, 2):
                vals.append(float(bf16_bits_to_f32(np.array([b + dlt], np.uint16))[0]))
            g = np.zeros(32, np.float32)
            g[0] = 127.0 * sc
            g[1:1 + len(vals)] = vals
            g[6:] = np.linspace(-126.0, 126.0, 26, dtype=np.float32) * sc
            groups.append(g)
    tiny = np.zeros(32, np.float32)
    tiny[:8] = np.float32(2.0 ** -130) * np.arange(1, 9, dtype=np.float32)   # subnormal scale
    tiny[8:16] = -tiny[:8]
    groups += [tiny, np.zeros(32, np.float32)]
    d = 128
    while len(groups) % (d // 32):
        groups.append(groups[0])
    x = np.stack(groups).reshape(1, -1, 1, d)                   # [B=1][T][Hkv=1][d]
    bits = to_bf16_bits(x)
    xf = bf16_bits_to_f32(bits)
    T = x.shape[1]
    S, W = 8, T + 8                                            # every token lands in the ring, in order
    cache = nd().KVCache.empty(1, 1, d, S, W)
    nd().nd_kv_cache_from_prefill(cache, dev_bf16(bits), dev_bf16(bits[:, ::-1].copy()),
                                  dev(np.zeros(1, np.int32)))
    wc, ws = oracle.quant_g32(xf[0, :, 0])
    vc, vs = oracle.quant_g32(xf[0, ::-1, 0])
    np.testing.assert_array_equal(host(cache.k_codes)[0, 0, S:S + T], wc)
    np.testing.assert_array_equal(host(cache.k_scale)[0, 0, S:S + T].view(np.uint32), ws.view(np.uint32))
    np.testing.assert_array_equal(host(cache.v_codes)[0, 0, S:S + T], vc)
    np.testing.assert_array_equal(host(cache.v_scale)[0, 0, S:S + T].view(np.uint32), vs.view(np.uint32))
    assert int(host(cache.ring_len)[0]) == T and int(host(cache.ring_start)[0]) == 0


def test_fill_rejections_and_scattered_segments():
    """Segment ids that repeat out of order (a segment's tokens are not one
    run), sink flags after the ring has started (rejected), sink prefixes
    longer than the sink region (rejected past sink_cap), a segment with no
    ring token, no seg_ids / no sink arrays, and invalid map entries."""
    rng = philox(3100)
    B, T, Hkv, d, S, W = 3, 333, 2, 64, 8, 40
    kb, kf = normal_bf16(rng, (B, T, Hkv, d))
    vb, vf = normal_bf16(rng, (B, T, Hkv, d))
    seg = np.empty((B, T), np.int32)
    seg[0] = 1 + (np.arange(T) // 7) % 5                  # five interleaved segments
    seg[1] = 1
    seg[1, 100:] = 2
    seg[1, 250:260] = 0                                   # padding inside segment 2
    seg[2] = 3
    sink = np.zeros((B, T), np.uint8)
    sink[0, ::3] = 1                                      # sinks everywhere: most rejected
    sink[1, :20] = 1                                      # prefix of 20 > S = 8 slots
    sink[1, 100:150] = 1                                  # segment 2: 50 sink tokens, no ring yet
    sink[1, 180] = 1                                      # a sink after segment 2's ring started
    sink[2, :] = 1                                        # a segment of sinks only
    entries = [(0, s) for s in range(1, 6)] + [(1, 1), (1, 2), (2, 3)]
    src_row = np.array([b for b, _ in entries], np.int32)
    src_seg = np.array([s for _, s in entries], np.int32)
    cache = nd().KVCache.empty(len(entries), Hkv, d, S, W)
    nd().nd_kv_cache_from_prefill(cache, dev_bf16(kb), dev_bf16(vb), dev(src_row), dev(seg), dev(sink),
                                  dev(src_seg))
    assert nd().nd_device_errors(clear=True) == 2          # rejected sink tokens are flagged
    ref, rejected = replay(kf, vf, seg, sink, entries, Hkv, d, S, W)
    assert min(rejected[:5]) > 0 and rejected[5] > 0 and rejected[7] > 0
    compare_filled(cache, ref, list(range(len(entries))))
    # no seg_ids, no sink: the whole batch row is one segment of ring tokens
    c2 = nd().KVCache.empty(B, Hkv, d, S, W)
    nd().nd_kv_cache_from_prefill(c2, dev_bf16(kb), dev_bf16(vb), dev(np.arange(B, dtype=np.int32)))
    ref2, rej2 = replay(kf, vf, None, None, [(b, 1) for b in range(B)], Hkv, d, S, W)
    assert sum(rej2) == 0
    compare_filled(c2, ref2, list(range(B)))
    # a batch row out of range and a padding segment id: flagged, untouched
    c3 = nd().KVCache.empty(2, Hkv, d, S, W)
    nd().nd_kv_cache_from_prefill(c3, dev_bf16(kb), dev_bf16(vb), dev(np.array([B, 0], np.int32)), dev(seg),
                                  dev(sink), dev(np.array([1, 0], np.int32)))
    assert nd().nd_device_errors(clear=True) == 2
    assert np.all(host(c3.seq_len) == 0) and np.all(host(c3.k_codes) == 0)


def test_fill_full_size_then_decode_step():
    """The packed-prefill workload at full size (B8 T4096 Hkv8 d128, every
    segment of every row, 512 sink slots + a 256-slot ring) handed to a cache,
    every row compared with the oracle replay; then one decode step
    (append + attend, Hq32, W256) on the filled cache against the oracle."""
    w = packed_prefill()
    B, T, Hq, d = w["q"].shape
    Hkv, S, W = w["k"].shape[2], 512, w["window"]
    seg, sink = w["seg_ids"], w["sink"]
    entries = [(b, int(s)) for b in range(B) for s in np.unique(seg[b]) if s > 0]
    src_row = np.array([b for b, _ in entries], np.int32)
    src_seg = np.array([s for _, s in entries], np.int32)
    n = len(entries)
    cache = nd().KVCache.empty(n, Hkv, d, S, W)
    nd().nd_kv_cache_from_prefill(cache, dev_bf16(w["k_bits"]), dev_bf16(w["v_bits"]), dev(src_row), dev(seg),
                                  dev(sink), dev(src_seg))
    ref, rejected = replay(w["k"], w["v"], seg, sink, entries, Hkv, d, S, W)
    assert sum(rejected) == 0
    compare_filled(cache, ref, list(range(n)))
    rng = philox(3200)
    kb, kf = normal_bf16(rng, (n, Hkv, d))
    vb, vf = normal_bf16(rng, (n, Hkv, d))
    qb, qf = normal_bf16(rng, (n, Hq, d))
    lse = torch.empty((n, Hq), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_decode_step(dev_bf16(qb), cache, dev_bf16(kb), dev_bf16(vb), W, lse=lse)
    oracle.kv_append(ref, kf, vf, False)
    want, wlse = oracle.decode(qf, ref, W)
    assert_close_bf16(host(out), want, "decode after handoff")
    np.testing.assert_allclose(host(lse), wlse, atol=2e-3, rtol=0)
