"""GPU parity: prefill attention under make_causal_packing_mask, rotary
embedding, block pooling with midpoint rotation and compressed attention,
against the fp64 oracle.  fp32 paths within 1e-4; bf16 outputs within max-abs
2e-2 / mean-abs 2e-3."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_close_bf16, assert_close_f32, dev, dev_bf16, host, need_gpu,
                      no_device_errors)
from workloads import (compressed, normal_bf16, packed_prefill, packed_segments, philox,
                       tiny_prefill)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    no_device_errors()


def nd():
    import sliding_window_kv_swa_gb300 as m
    return m


def oracle_rows(q, k, v, seg, sink, window, theta, rows):
    """Oracle prefill for sampled (b, t) rows: mask rows of one batch row at a
    time, rotation of q at the sampled positions and of k at every position."""
    out = np.empty((len(rows), q.shape[2], q.shape[3]))
    lse = np.empty((len(rows), q.shape[2]))
    for b in sorted(set(int(r[0]) for r in rows)):
        idx = [i for i, r in enumerate(rows) if r[0] == b]
        ts = np.array([rows[i][1] for i in idx])
        T = q.shape[1]
        qb = q[b, ts][None].astype(np.float64)
        kb = k[b:b + 1].astype(np.float64)
        if theta:
            qb = oracle.rope(qb, ts.astype(np.int64), theta)
            kb = oracle.rope(kb, np.arange(T), theta)
        mask = oracle.causal_packing_mask(seg[b:b + 1], None if sink is None else sink[b:b + 1], window)
        o, l = oracle.attention(qb, kb, v[b:b + 1], mask[:, ts])
        out[idx], lse[idx] = o[0], l[0]
    return out, lse


# ---------------------------------------------------------------- fp32

@pytest.mark.parametrize("single", [False, True])
def test_tiny_prefill_fp32(single):
    w = tiny_prefill(single_segment=single)
    lse = torch.empty((1, 4, 512), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_prefill(dev(w["q"]), dev(w["k"]), dev(w["v"]), dev(w["seg_ids"]), dev(w["sink"]),
                                   w["window"], lse=lse)
    want, wlse = oracle.swa_sink_prefill(w["q"], w["k"], w["v"], w["seg_ids"], w["sink"], w["window"])
    assert_close_f32(host(out), want, "tiny prefill")
    np.testing.assert_allclose(host(lse).transpose(0, 2, 1), wlse, atol=1e-4, rtol=0)


def test_fp32_variants():
    rng = philox(700)
    B, T, Hq, Hkv, d = 2, 333, 6, 2, 128
    q, k, v = (rng.standard_normal((B, T, H, d), dtype=np.float32) for H in (Hq, Hkv, Hkv))
    seg, sink = packed_segments(rng, B, T, 2, 3, 40, 5, 30)
    seg[1, 300:] = 0                                  # padding tail
    for window, theta, use_sink in ((0, 0.0, False), (17, 0.0, True), (64, 10000.0, True)):
        s = sink if use_sink else None
        out = nd().nd_swa_sink_prefill(dev(q), dev(k), dev(v), dev(seg), None if s is None else dev(s),
                                       window, rope_theta=theta)
        want, _ = oracle.swa_sink_prefill(q, k, v, seg, s, window, theta)
        assert_close_f32(host(out), want, f"fp32 W={window} theta={theta}")


def test_fp32_unsplit():
    """Above 256 CTAs of 16 rows the fp32 kernel keeps each row tile's keys in
    one CTA (smaller problems split them over four and merge): B2 T700 Hq8
    (704 CTAs), packed segments with sinks, a window."""
    rng = philox(710)
    B, T, Hq, Hkv, d = 2, 700, 8, 2, 64
    q, k, v = (rng.standard_normal((B, T, H, d), dtype=np.float32) for H in (Hq, Hkv, Hkv))
    seg, sink = packed_segments(rng, B, T, 2, 4, 60, 5, 40)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_prefill(dev(q), dev(k), dev(v), dev(seg), dev(sink), 100, lse=lse)
    want, wlse = oracle.swa_sink_prefill(q, k, v, seg, sink, 100)
    assert_close_f32(host(out), want, "fp32 unsplit")
    np.testing.assert_allclose(host(lse).transpose(0, 2, 1), wlse, atol=1e-4, rtol=0)


# ---------------------------------------------------------------- bf16

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T,Hq,Hkv,window", [(1, 2, 1, 256), (200, 4, 4, 32), (517, 8, 2, 100),
                                             (1000, 4, 1, 256), (700, 3, 1, 0)])
def test_bf16_packed_small(d, T, Hq, Hkv, window):
    rng = philox(800 + T + d)
    B = 2
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    if T >= 200:
        seg, sink = packed_segments(rng, B, T, 2, 3, T // 4, 3, T // 8)
    else:
        seg = np.ones((B, T), np.int32)
        sink = np.zeros((B, T), np.uint8)
        sink[:, :3] = 1
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink), window,
                                   rope_theta=10000.0, lse=lse)
    want, wlse = oracle.swa_sink_prefill(q, k, v, seg, sink, window, 10000.0)
    assert_close_bf16(host(out), want, f"bf16 T={T}")
    np.testing.assert_allclose(host(lse).transpose(0, 2, 1), wlse, atol=2e-2, rtol=0)


def test_bf16_padding_rows_are_zero():
    rng = philox(900)
    B, T, Hq, Hkv, d = 1, 300, 4, 2, 64
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    seg = np.ones((B, T), np.int32)
    seg[0, 100:180] = 0
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    out = host(nd().nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), None, 64, lse=lse))
    assert np.all(out[0, 100:180] == 0)
    assert np.all(np.isneginf(host(lse)[0, :, 100:180]))
    want, _ = oracle.swa_sink_prefill(q, k, v, seg, None, 64)
    assert_close_bf16(out, want, "padding")


@pytest.mark.parametrize("window", [0, 256])
def test_bf16_zero_gap_inside_segment(window):
    """Keys with segment id 0 between two runs of the same id are never
    visible, also to whole warps of later rows that see their tile entirely
    (causal bound and window), where the per-tile fast path applies."""
    rng = philox(910 + window)
    B, T, Hq, Hkv, d = 1, 640, 4, 2, 128
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    seg = np.ones((B, T), np.int32)
    seg[0, 100:180] = 0
    sink = np.zeros((B, T), np.uint8)
    sink[0, [5, 64, 130, 200]] = 1
    out = host(nd().nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink), window))
    want, _ = oracle.swa_sink_prefill(q, k, v, seg, sink, window)
    assert_close_bf16(out, want, f"zero gap W={window}")


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (3, 1, 64)])
def test_bf16_empty_spans(Hq, Hkv, d):
    """Row spans with no visible key at all (segment id 0 over whole 128-row
    blocks, in the middle and at the end): their work items have no tiles,
    output 0 and lse -inf, and the items after them (sharing the persistent
    CTAs' barrier phases and O buffers) stay exact."""
    rng = philox(930 + d)
    B, T = 2, 1000
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    seg = np.ones((B, T), np.int32)
    seg[0, 256:512] = 0          # two whole 128-row blocks
    seg[0, 512:] = 2             # then a new segment
    seg[1, 640:] = 0             # a padded tail, including the ragged last block
    sink = np.zeros((B, T), np.uint8)
    sink[:, :8] = 1
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    out = host(nd().nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink), 128,
                                        lse=lse))
    assert np.all(out[0, 256:512] == 0) and np.all(out[1, 640:] == 0)
    assert np.all(np.isneginf(host(lse)[0, :, 256:512]))
    want, wlse = oracle.swa_sink_prefill(q, k, v, seg, sink, 128)
    assert_close_bf16(out, want, "empty spans")
    got_lse = host(lse).transpose(0, 2, 1)
    fin = np.isfinite(wlse)
    assert np.array_equal(fin, np.isfinite(got_lse))
    np.testing.assert_allclose(got_lse[fin], wlse[fin], atol=2e-2, rtol=0)


def test_bf16_many_segments_per_tile():
    """Tiles holding more than four segment ids (short segments, ids
    repeating out of order) and tiles holding two to four."""
    rng = philox(920)
    B, T, Hq, Hkv, d = 2, 512, 4, 2, 64
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    seg = np.empty((B, T), np.int32)
    seg[0] = 1 + (np.arange(T) // 6) % 9          # runs of 6: up to 11 ids per 64-key tile
    seg[1] = 1 + (np.arange(T) // 24)             # runs of 24: 3 or 4 ids per tile
    seg[1, 300:310] = 0
    sink = (philox(921).random((B, T)) < 0.05).astype(np.uint8)
    for window in (0, 40):
        out = host(nd().nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink),
                                            window))
        want, _ = oracle.swa_sink_prefill(q, k, v, seg, sink, window)
        assert_close_bf16(out, want, f"many segments W={window}")


def test_packed_prefill_full_size_planes():
    """Packed-segment prefill at full size (B8 T4096 Hq32 Hkv8 d128, W256,
    RoPE) in the bench's launch configuration.  Batch rows 0 and 7 are
    compared whole (every row and head, out and lse) with the oracle, so every
    persistent work item of those rows -- and the barrier phases each CTA
    carries from one item to the next -- is checked; the other rows on their
    first and last positions, around segment starts and at random."""
    w = packed_prefill()
    B, T, Hq, d = w["q"].shape
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_prefill(dev_bf16(w["q_bits"]), dev_bf16(w["k_bits"]), dev_bf16(w["v_bits"]),
                                   dev(w["seg_ids"]), dev(w["sink"]), w["window"], rope_theta=w["rope_theta"],
                                   lse=lse)
    got, got_lse = host(out), host(lse)
    rows = [(b, t) for b in (0, B - 1) for t in range(T)]
    rng = philox(901)
    for b in range(1, B - 1):
        rows += [(b, 0), (b, T - 1)] + [(b, int(t)) for t in rng.integers(0, T, size=24)]
        starts = np.nonzero(np.diff(w["seg_ids"][b]))[0] + 1
        for s0 in starts:
            rows += [(b, int(s0)), (b, int(s0) - 1), (b, min(int(s0) + 300, T - 1))]
    want, wlse = oracle_rows(w["q"], w["k"], w["v"], w["seg_ids"], w["sink"], w["window"], w["rope_theta"], rows)
    gr = np.stack([got[b, t] for b, t in rows])
    assert_close_bf16(gr, want, "packed prefill rows")
    gl = np.stack([got_lse[b, :, t] for b, t in rows])
    np.testing.assert_allclose(gl, wlse, atol=2e-2, rtol=0)
    for b in (0, B - 1):   # each whole plane on its own as well
        sel = [i for i, r in enumerate(rows) if r[0] == b]
        assert_close_bf16(gr[sel], want[sel], f"packed prefill batch row {b}")


# ---------------------------------------------------------------- rope / pool / compressed

@pytest.mark.parametrize("d", [64, 128])
def test_rope_matches_oracle(d):
    rng = philox(1000 + d)
    B, T, H = 2, 4096, 3
    xb, x = normal_bf16(rng, (B, T, H, d))
    y = host(nd().nd_rope_apply(dev_bf16(xb), rope_theta=10000.0))
    want = oracle.rope(x, np.arange(T), 10000.0)
    err = np.abs(y - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3      # bf16 output rounding
    assert np.all(err <= np.abs(want) * 2 ** -8 + 1e-6)   # one bf16 rounding per element


@pytest.mark.parametrize("block,T,d", [(4, 4096, 64), (1, 100, 64), (3, 101, 64), (8, 64, 64), (4, 1000, 128),
                                       (5, 203, 48), (64, 4096, 64), (2, 50, 62), (1, 8192, 64)])
def test_compress_pool_matches_oracle(block, T, d):
    # d = 62 (not a multiple of 16) takes the scalar pooling kernel, the rest
    # the 16-byte one; T % block leaves a dropped tail in several cases
    rng = philox(1100 + block + d)
    B, H = 2, 4
    kb, k = normal_bf16(rng, (B, T, H, d))
    vb, v = normal_bf16(rng, (B, T, H, d))
    pk, pv = nd().nd_kv_compress_pool(dev_bf16(kb), dev_bf16(vb), block, 10000.0)
    _, kk, vv = oracle.compress(k, k, v, block, 10000.0)
    nb = T // block
    for got, want, name in ((host(pk), kk[:, :nb], "pooled k"), (host(pv), vv[:, :nb], "pooled v")):
        err = np.abs(got - want)
        assert np.all(err <= np.abs(want) * 2 ** -8 + 1e-6), name


def test_compressed_prefill_full_size():
    """Compressed-attention configuration at full size (B4 T4096 H16 d64, W256,
    b4, RoPE): pool (GPU) + rotation + attention.  Batch row 0 is compared
    whole (every row and head) with the oracle; the other rows at the window
    edge and block-arrival rows (255-263), the last row and at random."""
    w = compressed()
    B, T, H, d = w["q"].shape
    pk, pv = nd().nd_kv_compress_pool(dev_bf16(w["k_bits"]), dev_bf16(w["v_bits"]), w["block"], w["rope_theta"])
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_prefill(dev_bf16(w["q_bits"]), dev_bf16(w["k_bits"]), dev_bf16(w["v_bits"]),
                                   None, None, w["window"], rope_theta=w["rope_theta"], pooled_k=pk,
                                   pooled_v=pv, block=w["block"], lse=lse)
    got, got_lse = host(out), host(lse)
    rng = philox(1200)
    rows = [(0, t) for t in range(T)]
    rows += [(b, t) for b in range(1, B) for t in (0, 255, 256, 258, 259, 262, 263, 1000, T - 1)]
    rows += [(int(rng.integers(1, B)), int(rng.integers(0, T))) for _ in range(64)]
    rows = np.array(rows)
    want, wlse = oracle.compressed_prefill(w["q"], w["k"], w["v"], w["window"], w["block"], w["rope_theta"],
                                           rows=rows)
    gr = np.stack([got[b, t] for b, t in rows])
    assert_close_bf16(gr, want, "compressed rows")
    assert_close_bf16(gr[:T], want[:T], "compressed batch row 0")
    np.testing.assert_allclose(np.stack([got_lse[b, :, t] for b, t in rows]), wlse, atol=2e-2, rtol=0)


@pytest.mark.parametrize("T,W,block", [(300, 16, 4), (129, 1, 2), (513, 64, 8), (64, 8, 1)])
def test_compressed_prefill_small_all_rows(T, W, block):
    rng = philox(1300 + T)
    B, H, d = 2, 4, 64
    qb, q = normal_bf16(rng, (B, T, H, d))
    kb, k = normal_bf16(rng, (B, T, H, d))
    vb, v = normal_bf16(rng, (B, T, H, d))
    pk, pv = nd().nd_kv_compress_pool(dev_bf16(kb), dev_bf16(vb), block, 10000.0)
    out = nd().nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), None, None, W, rope_theta=10000.0,
                                   pooled_k=pk, pooled_v=pv, block=block)
    want, _ = oracle.compressed_prefill(q, k, v, W, block, 10000.0)
    assert_close_bf16(host(out), want, f"compressed T={T}")


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 1)])
def test_bf16_rotation_in_kernel_matches_separate_rope(d, Hq, Hkv):
    # q is rotated inside the attention kernel as its tile is staged; the
    # result must carry the same bits as rotating q and k with the stand-alone
    # rotary call and running the product without rotation.  T spans a ragged
    # last row block; (3, 1) takes the unpaired-head path (two row blocks).
    rng = philox(1700 + d + Hq)
    B, T, W = 2, 389, 96
    qb, _ = normal_bf16(rng, (B, T, Hq, d))
    kb, _ = normal_bf16(rng, (B, T, Hkv, d))
    vb, _ = normal_bf16(rng, (B, T, Hkv, d))
    seg, sink = packed_segments(rng, B, T, 2, 3, T // 4, 3, T // 8)
    lib = nd()
    fused = lib.nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink), W,
                                    rope_theta=10000.0)
    qr = lib.nd_rope_apply(dev_bf16(qb), rope_theta=10000.0)
    kr = lib.nd_rope_apply(dev_bf16(kb), rope_theta=10000.0)
    sep = lib.nd_swa_sink_prefill(qr, kr, dev_bf16(vb), dev(seg), dev(sink), W, rope_theta=0.0)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), sep.view(torch.int16))


@pytest.mark.gpu
def test_prefill_calls_back_to_back_share_a_workspace():
    """Prefill calls enqueued back to back on one workspace with no
    synchronisation (each call's tile records, angle table, rotated K and the
    attention kernel are chained dependent launches): every output must carry
    the same bits as the same call run alone."""
    rng = philox(1800)
    lib = nd()
    B, T, Hq, Hkv, d = 2, 700, 4, 2, 128
    calls = []
    for i in range(3):
        qb, _ = normal_bf16(rng, (B, T, Hq, d))
        kb, _ = normal_bf16(rng, (B, T, Hkv, d))
        vb, _ = normal_bf16(rng, (B, T, Hkv, d))
        seg, sink = packed_segments(rng, B, T, 2, 3, T // 4, 3, T // 8)
        calls.append((dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink), [64, 17, 256][i],
                      [10000.0, 0.0, 500000.0][i]))
    nbytes = max(lib.nd_swa_sink_prefill_workspace_size(lib.ND_BF16, B, T, Hq, Hkv, d, th, 0)
                 for *_, th in calls)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    alone = []
    for q, k, v, seg, sink, W, th in calls:
        alone.append(lib.nd_swa_sink_prefill(q, k, v, seg, sink, W, rope_theta=th, workspace=ws))
        torch.cuda.synchronize()
    chained = [torch.empty_like(a) for a in alone]
    for (q, k, v, seg, sink, W, th), o in zip(calls, chained):
        lib.nd_swa_sink_prefill(q, k, v, seg, sink, W, rope_theta=th, out=o, workspace=ws)
    torch.cuda.synchronize()
    for i, (a, c) in enumerate(zip(alone, chained)):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16)), f"call {i}"


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 64), (3, 1, 128)])
def test_prefill_tile_count_reported_by_the_kernel_plan(Hq, Hkv, d):
    """nd_swa_sink_prefill_tiles reads the plan the call built: at least
    every (128-row block, 64-key tile) holding a visible pair (brute force on
    the oracle's mask) times the query heads, at most every causal tile of
    the span the plan covers; one segment without sinks or window: exactly
    the causal tiles."""
    rng = philox(1900 + d)
    B, T, W = 2, 700, 100
    qb, _ = normal_bf16(rng, (B, T, Hq, d))
    kb, _ = normal_bf16(rng, (B, T, Hkv, d))
    vb, _ = normal_bf16(rng, (B, T, Hkv, d))
    seg, sink = packed_segments(rng, B, T, 2, 4, 120, 3, 40)
    lib = nd()
    pair = (Hq // Hkv) % 2 == 0
    span = 128 if pair else 256
    blocks = 1 if pair else 2
    for segs, snk, win in ((seg, sink, W), (np.ones((B, T), np.int32), None, 0)):
        ws = torch.empty(lib.nd_swa_sink_prefill_workspace_size(lib.ND_BF16, B, T, Hq, Hkv, d, 0.0, 0),
                         dtype=torch.uint8, device="cuda")
        lib.nd_swa_sink_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(segs),
                                None if snk is None else dev(snk), win, workspace=ws)
        got = lib.nd_swa_sink_prefill_tiles(ws, B, T, Hq, Hkv, d, 0.0, 0)
        mask = oracle.causal_packing_mask(segs, snk, win)
        visible = causal = 0
        for b in range(B):
            for q0 in range(0, T, 128):
                q1 = min(T, q0 + 128)
                visible += sum(bool(mask[b, q0:q1, k0:k0 + 64].any()) for k0 in range(0, q1, 64))
            for q0 in range(0, T, span):
                causal += ((min(T, q0 + span) - 1) // 64 + 1) * blocks
        assert visible * Hq <= got <= causal * Hq, (visible * Hq, got, causal * Hq)
        if snk is None:
            assert got == causal * Hq


@pytest.mark.parametrize("block,T,d,theta", [(4, 4096, 64, 10000.0), (3, 301, 64, 10000.0), (8, 1000, 128, 500000.0),
                                             (1, 77, 64, 10000.0), (4, 258, 128, 0.0), (16, 10, 64, 10000.0),
                                             (64, 300, 64, 10000.0)])
def test_pool_rope_pass_matches_the_separate_passes(block, T, d, theta):
    """nd_kv_compress_pool_rope (one read of K and V) gives bit for bit the
    rotated keys of nd_rope_apply and the pooled blocks of nd_kv_compress_pool
    (positions past the last whole block are rotated too).  The cases cover
    both forms of the pass: chunks of whole blocks moved by bulk copies, and
    the per-thread form for a pooled block of more than 16 KB (block 64 here)
    or a sequence shorter than one block."""
    rng = philox(1950 + block + T + d)
    B, H = 2, 3
    kb, _ = normal_bf16(rng, (B, T, H, d))
    vb, _ = normal_bf16(rng, (B, T, H, d))
    lib = nd()
    k_d, v_d = dev_bf16(kb), dev_bf16(vb)
    k_rot, pk, pv = lib.nd_kv_compress_pool_rope(k_d, v_d, block, theta)
    rk, rv = lib.nd_kv_compress_pool(k_d, v_d, block, theta)
    torch.cuda.synchronize()
    assert torch.equal(pk.view(torch.int16), rk.view(torch.int16))
    assert torch.equal(pv.view(torch.int16), rv.view(torch.int16))
    if theta:
        assert torch.equal(k_rot.view(torch.int16), lib.nd_rope_apply(k_d, rope_theta=theta).view(torch.int16))


@pytest.mark.parametrize("T,W,block,d,H", [(4096, 256, 4, 64, 16), (700, 40, 8, 128, 4), (301, 17, 3, 64, 2),
                                           (129, 1, 2, 128, 3)])
def test_compressed_prefill_pooling_inside_the_call(T, W, block, d, H):
    """With pooled_k = pooled_v = NULL the compressed prefill pools K and V
    itself in the same pass that rotates K: the output carries the same bits
    as pooling with nd_kv_compress_pool first (and matches the oracle)."""
    rng = philox(1960 + T + d)
    B = 2 if T < 4096 else 1
    qb, q = normal_bf16(rng, (B, T, H, d))
    kb, k = normal_bf16(rng, (B, T, H, d))
    vb, v = normal_bf16(rng, (B, T, H, d))
    lib = nd()
    q_d, k_d, v_d = dev_bf16(qb), dev_bf16(kb), dev_bf16(vb)
    pk, pv = lib.nd_kv_compress_pool(k_d, v_d, block, 10000.0)
    lse_a = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    lse_b = torch.empty_like(lse_a)
    a = lib.nd_swa_sink_prefill(q_d, k_d, v_d, None, None, W, rope_theta=10000.0, pooled_k=pk, pooled_v=pv,
                                block=block, lse=lse_a)
    b = lib.nd_swa_sink_prefill(q_d, k_d, v_d, None, None, W, rope_theta=10000.0, block=block, lse=lse_b)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)
    if T < 4096:
        want, _ = oracle.compressed_prefill(q, k, v, W, block, 10000.0)
        assert_close_bf16(host(b), want, "pooling inside the call")


@pytest.mark.parametrize("T,W,block,P,d,H", [(300, 16, 4, 5, 64, 4), (513, 40, 8, 64, 128, 2), (129, 1, 2, 0, 64, 3),
                                             (700, 64, 4, 100, 64, 4), (200, 30, 3, 200, 128, 2),
                                             (4096, 256, 4, 512, 64, 16)])
def test_compressed_prefill_with_pinned_prefix(T, W, block, P, d, H):
    """nd_compressed_prefill: the first P keys pinned (visible at any
    distance), pooled blocks over the positions after them, the exact window;
    every row (the 4096-token case: every row of the one sequence) against
    the oracle; without pins, the same bits as the compressed
    nd_swa_sink_prefill."""
    rng = philox(1990 + T + P + d)
    B = 2 if T < 4096 else 1
    qb, q = normal_bf16(rng, (B, T, H, d))
    kb, k = normal_bf16(rng, (B, T, H, d))
    vb, v = normal_bf16(rng, (B, T, H, d))
    lib = nd()
    q_d, k_d, v_d = dev_bf16(qb), dev_bf16(kb), dev_bf16(vb)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    out = lib.nd_compressed_prefill(q_d, k_d, v_d, W, block, n_pinned=P, rope_theta=10000.0, lse=lse)
    want, wlse = oracle.compressed_prefill_pinned(q, k, v, W, block, P, 10000.0)
    assert_close_bf16(host(out), want, f"pinned {P}")
    np.testing.assert_allclose(host(lse).transpose(0, 2, 1), wlse, atol=2e-2, rtol=0)
    if P == 0:
        ref = lib.nd_swa_sink_prefill(q_d, k_d, v_d, None, None, W, rope_theta=10000.0, block=block)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
