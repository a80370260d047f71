"""Pins for the oracle's dense attention, codec, cache and decode (CPU only).

Attention is checked against torch's scaled_dot_product_attention in float64
(a library routine: plain causal, GQA by repeat_interleave, explicit boolean
masks), a two-key case worked by hand, and the sink invariants the Needle pages
state.  The codec is checked against hand-derived codes; the ring cache against
a deque simulation; decode against the prefill mask's last row.
"""
import collections
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_path
from workloads import bf16_bits_to_f32, decode_cache, philox, tiny_prefill, to_bf16_bits


def sdpa(q, k, v, mask=None, causal=False):
    """torch SDPA in float64 on [B,T,H,d] arrays (GQA via repeat_interleave)."""
    G = q.shape[2] // k.shape[2]
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    m = None if mask is None else torch.from_numpy(mask)[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, is_causal=causal)
    return o.permute(0, 2, 1, 3).numpy()


def rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 1), (8, 2), (6, 3)])
def test_wide_window_reduces_to_causal_sdpa(Hq, Hkv):
    rng = philox(11)
    B, T, d = 2, 37, 16
    q, k, v = rand(rng, B, T, Hq, d), rand(rng, B, T, Hkv, d), rand(rng, B, T, Hkv, d)
    seg = np.ones((B, T), np.int32)
    out, _ = oracle.swa_sink_prefill(q, k, v, seg, None, window=T)
    np.testing.assert_allclose(out, sdpa(q, k, v, causal=True), rtol=0, atol=1e-12)


def test_masked_attention_matches_sdpa_with_mask():
    rng = philox(12)
    B, T, Hq, Hkv, d = 2, 29, 4, 2, 8
    q, k, v = rand(rng, B, T, Hq, d), rand(rng, B, T, Hkv, d), rand(rng, B, T, Hkv, d)
    seg = np.repeat(np.array([[1] * 10 + [2] * 19, [3] * 29]), 1, 0).astype(np.int32)
    sink = (rng.random((B, T)) < 0.2).astype(np.uint8)
    mask = oracle.causal_packing_mask(seg, sink, 5)
    out, lse = oracle.attention(q, k, v, mask)
    np.testing.assert_allclose(out, sdpa(q, k, v, mask=mask), rtol=0, atol=1e-12)
    # lse is log of the softmax denominator: recompute it from raw scores
    G = Hq // Hkv
    for b, t, h in [(0, 3, 1), (1, 28, 3), (0, 20, 0)]:
        s = q[b, t, h] @ k[b, :, h // G].T / math.sqrt(d)
        want = np.log(np.exp(s[mask[b, t]]).sum())
        assert abs(lse[b, t, h] - want) < 1e-12


def test_two_keys_by_hand():
    # d = 2, q = (1, 0); keys (0, 0) and (2, 0) give scores 0 and 2/sqrt(2);
    # values (1, 0) and (0, 1): out = (1 - p, p), p = e^r / (1 + e^r), r = sqrt(2).
    q = np.array([[[[1.0, 0.0]], [[1.0, 0.0]]]])
    k = np.array([[[[0.0, 0.0]], [[2.0, 0.0]]]])
    v = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    out, lse = oracle.swa_sink_prefill(q, k, v, np.ones((1, 2), np.int32), None, 0)
    r = math.sqrt(2.0)
    p = math.exp(r) / (1 + math.exp(r))
    np.testing.assert_allclose(out[0, 1, 0], [1 - p, p], atol=1e-15)
    assert abs(lse[0, 1, 0] - math.log(1 + math.exp(r))) < 1e-14
    np.testing.assert_allclose(out[0, 0, 0], [1.0, 0.0], atol=0)  # row 0 sees only key 0


def test_fully_masked_row_is_zero_not_nan():
    rng = philox(13)
    q, k, v = rand(rng, 1, 4, 2, 8), rand(rng, 1, 4, 1, 8), rand(rng, 1, 4, 1, 8)
    seg = np.array([[1, 0, 1, 1]], np.int32)
    out, lse = oracle.swa_sink_prefill(q, k, v, seg, None, 2)
    assert np.all(out[0, 1] == 0) and np.all(np.isneginf(lse[0, 1]))
    assert np.all(np.isfinite(out))


def test_rows_subset_matches_full():
    w = tiny_prefill(single_segment=True)
    full, lse = oracle.swa_sink_prefill(w["q"], w["k"], w["v"], w["seg_ids"], w["sink"], w["window"])
    rows = np.array([[0, 0], [0, 47], [0, 300], [0, 511]])
    sub, lse_s = oracle.swa_sink_prefill(w["q"], w["k"], w["v"], w["seg_ids"], w["sink"], w["window"], rows=rows)
    np.testing.assert_array_equal(sub, full[0, rows[:, 1]])
    np.testing.assert_array_equal(lse_s, lse[0, rows[:, 1]])


def test_sink_perturbation_reaches_far_rows():
    w = tiny_prefill(single_segment=True)
    base, _ = oracle.swa_sink_prefill(w["q"], w["k"], w["v"], w["seg_ids"], w["sink"], w["window"])
    v2 = w["v"].copy()
    v2[0, 0] += 1.0          # a sink value, 511 positions before the last row
    pert, _ = oracle.swa_sink_prefill(w["q"], w["k"], v2, w["seg_ids"], w["sink"], w["window"])
    assert np.abs(pert[0, 511] - base[0, 511]).max() > 1e-6
    v3 = w["v"].copy()
    v3[0, 100] += 1.0        # a non-sink value outside row 511's window
    pert3, _ = oracle.swa_sink_prefill(w["q"], w["k"], v3, w["seg_ids"], w["sink"], w["window"])
    np.testing.assert_array_equal(pert3[0, 511], base[0, 511])
    # the literal two-segment layout: seg-2 rows never see the seg-1 sinks
    w2 = tiny_prefill(single_segment=False)
    b2, _ = oracle.swa_sink_prefill(w2["q"], w2["k"], w2["v"], w2["seg_ids"], w2["sink"], w2["window"])
    p2, _ = oracle.swa_sink_prefill(w2["q"], w2["k"], v2, w2["seg_ids"], w2["sink"], w2["window"])
    np.testing.assert_array_equal(p2[0, 48:], b2[0, 48:])


# ----------------------------------------------------------------------------
# codec
# ----------------------------------------------------------------------------

def read_codec_fixture():
    groups, cur = [], None
    for line in open(golden_path("codec_g32.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("group"):
            cur = {}
            groups.append(cur)
        else:
            key, vals = line.split(":", 1)
            cur[key] = [float(x) for x in vals.split()]
    return groups


def test_codec_hand_cases():
    groups = read_codec_fixture()
    x = np.array([g["x"] for g in groups], np.float32).reshape(1, -1)   # d = 128
    codes, scales = oracle.quant_g32(x)
    np.testing.assert_array_equal(codes.reshape(-1), np.array([g["code"] for g in groups]).reshape(-1).astype(np.int8))
    np.testing.assert_array_equal(scales.reshape(-1), np.array([g["scale"][0] for g in groups], np.float32))


def test_codec_properties_on_bf16_normals():
    rng = philox(21)
    bits = to_bf16_bits(rng.standard_normal((500, 128), dtype=np.float32) * rng.uniform(0.01, 100, (500, 1)).astype(np.float32))
    x = bf16_bits_to_f32(bits)
    codes, scales = oracle.quant_g32(x)
    xg = x.reshape(500, 4, 32)
    cg = codes.reshape(500, 4, 32).astype(np.int64)
    amax = np.abs(xg).max(-1)
    # the absmax element maps to +-127 and carries the sign of x
    idx = np.abs(xg).argmax(-1)
    top = np.take_along_axis(cg, idx[..., None], -1)[..., 0]
    top_x = np.take_along_axis(xg, idx[..., None], -1)[..., 0]
    assert np.all(np.abs(top) == 127) and np.all(np.sign(top) == np.sign(top_x))
    assert np.all(np.abs(cg) <= 127)
    # scale ~ amax / 127 (one fp32 rounding)
    np.testing.assert_allclose(scales, amax / 127.0, rtol=1e-7)
    # round trip error at most half a step (plus fp32 rounding of the quotient)
    err = np.abs(xg - cg * scales[..., None].astype(np.float64))
    assert np.all(err <= scales[..., None] * (0.5 + 1e-5))


def test_codec_zero_group():
    x = np.zeros((2, 64), np.float32)
    x[1, 40] = -3.0
    codes, scales = oracle.quant_g32(x)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0)
    assert scales[1, 0] == 0 and np.all(codes[1, :32] == 0)
    assert codes[1, 40] == -127


# ----------------------------------------------------------------------------
# ring cache and decode
# ----------------------------------------------------------------------------

def test_ring_append_matches_deque_simulation():
    rng = philox(31)
    B, Hkv, d, S, W = 3, 2, 32, 4, 5
    cache = oracle.Cache(B, Hkv, d, S, W)
    rings = [collections.deque(maxlen=W) for _ in range(B)]
    sinks = [[] for _ in range(B)]
    tokens = {}
    for step in range(3 + 17):
        to_sink = step < 3
        kt = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        vt = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        rej = oracle.kv_append(cache, kt, vt, to_sink)
        assert rej == 0
        for b in range(B):
            (sinks[b] if to_sink else rings[b]).append(step)
            tokens[(b, step)] = (kt[b], vt[b])
    # a sink append after ring tokens is rejected (the sink is a prefix)
    probe = cache.copy()
    assert oracle.kv_append(probe, kt, vt, True) == B
    np.testing.assert_array_equal(probe.k_codes, cache.k_codes)
    for b in range(B):
        kpos, is_sink = oracle.slot_positions(cache, b)
        assert list(kpos[:S][is_sink[:S]]) == sinks[b]
        assert sorted(kpos[S:][kpos[S:] >= 0]) == list(rings[b])
        assert cache.seq_len[b] == 20
        for s in range(S + W):
            if kpos[s] < 0:
                continue
            kt_, vt_ = tokens[(b, int(kpos[s]))]
            c, sc = oracle.quant_g32(kt_)
            np.testing.assert_array_equal(cache.k_codes[b, :, s], c)
            np.testing.assert_array_equal(cache.k_scale[b, :, s], sc)
            c, sc = oracle.quant_g32(vt_)
            np.testing.assert_array_equal(cache.v_codes[b, :, s], c)


def fill_cache(w, S, W):
    B, Hkv, ns, d = w["k"].shape
    cache = oracle.Cache(B, Hkv, d, S, W)
    cache.k_codes[...], cache.k_scale[...] = oracle.quant_g32(w["k"])
    cache.v_codes[...], cache.v_scale[...] = oracle.quant_g32(w["v"])
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        getattr(cache, f)[...] = w[f]
    return cache


@pytest.mark.parametrize("full", [True, False])
def test_decode_equals_prefill_last_row(full):
    # Lay the cached keys out by absolute position and run the prefill mask
    # (one segment, sinks = the prefix, same window): its last row must equal
    # the decode result.  Ties the decode mask to make_causal_packing_mask.
    S, W, Hq, Hkv, d = 6, 16, 4, 2, 32
    w = decode_cache(3, Hq, Hkv, d, S, W, seed=41, full=full)
    cache = fill_cache(w, S, W)
    out, lse = oracle.decode(w["q"], cache, window=W)
    for b in range(3):
        kpos, is_sink = oracle.slot_positions(cache, b)
        T = int(cache.seq_len[b])
        kd = np.zeros((1, T, Hkv, d))
        vd = np.zeros((1, T, Hkv, d))
        occupied = np.zeros(T, bool)
        for s in np.nonzero(kpos >= 0)[0]:
            kd[0, kpos[s]] = oracle.dequant_g32(cache.k_codes[b, :, s], cache.k_scale[b, :, s])
            vd[0, kpos[s]] = oracle.dequant_g32(cache.v_codes[b, :, s], cache.v_scale[b, :, s])
            occupied[kpos[s]] = True
        sink = np.zeros((1, T), np.uint8)
        sink[0, :S] = 1
        # positions evicted from the ring are outside the window anyway
        assert occupied[:S].all() and occupied[T - min(W, T - S):].all()
        qf = np.zeros((1, T, Hq, d))
        qf[0, T - 1] = w["q"][b]
        o, l = oracle.swa_sink_prefill(qf, kd, vd, np.ones((1, T), np.int32), sink, W,
                                       rows=np.array([[0, T - 1]]))
        np.testing.assert_allclose(out[b], o[0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse[b], l[0], atol=1e-12, rtol=0)


def test_decode_invariant_to_ring_rotation():
    S, W, Hq, Hkv, d = 4, 8, 2, 1, 32
    w = decode_cache(1, Hq, Hkv, d, S, W, seed=43, full=True)
    cache = fill_cache(w, S, W)
    out0, _ = oracle.decode(w["q"], cache, W)
    for shift in range(1, W):
        c2 = cache.copy()
        ring = slice(S, S + W)
        for arr in (c2.k_codes, c2.v_codes, c2.k_scale, c2.v_scale):
            arr[:, :, ring] = np.roll(arr[:, :, ring], shift, axis=2)
        c2.ring_start[0] = (cache.ring_start[0] + shift) % W
        out, _ = oracle.decode(w["q"], c2, W)
        np.testing.assert_allclose(out, out0, atol=1e-13, rtol=0)


def test_decode_window_smaller_than_ring_hides_oldest():
    S, W, Hq, Hkv, d = 2, 8, 1, 1, 32
    w = decode_cache(1, Hq, Hkv, d, S, W, seed=44, full=True)
    cache = fill_cache(w, S, W)
    out_full, _ = oracle.decode(w["q"], cache, W)
    out_w3, _ = oracle.decode(w["q"], cache, 3)
    assert np.abs(out_full - out_w3).max() > 1e-6
    # window 3 == attending over the sinks and the newest three ring slots only
    kpos, _ = oracle.slot_positions(cache, 0)
    newest = int(cache.seq_len[0]) - 1
    keep = [s for s in range(S + W) if s < S or newest - kpos[s] < 3]
    assert len(keep) == S + 3
    kd = oracle.dequant_g32(cache.k_codes[0, :, keep], cache.k_scale[0, :, keep])
    vd = oracle.dequant_g32(cache.v_codes[0, :, keep], cache.v_scale[0, :, keep])
    o, _ = oracle.attention(w["q"][:, None], kd[None], vd[None], np.ones((1, len(keep)), bool))
    np.testing.assert_allclose(out_w3[0], o[0, 0], atol=1e-13, rtol=0)


# ---------------------------------------------------------------- chunked prefill against the cache

def _exact_int8_tokens(rng, shape):
    """Token values the int8 group-32 codec stores exactly: per 32-channel
    group, codes in [-127, 127] with one at +-127, times 2^-6 (so
    amax/127 = 2^-6 and every x / scale is the integer code)."""
    codes = rng.integers(-127, 128, size=shape).astype(np.float64)
    g = codes.reshape(shape[:-1] + (shape[-1] // 32, 32))
    g[..., 0] = np.where(rng.random(g.shape[:-1]) < 0.5, 127.0, -127.0)
    return g.reshape(shape) / 64.0


@pytest.mark.parametrize("S,W,ring_cap,Tc,n_sink,n_before", [
    (8, 6, 6, 10, 5, 20),    # ring wrapped, window = ring
    (4, 5, 9, 7, 4, 3),      # ring partly filled, window < ring
    (6, 4, 4, 3, 0, 0),      # empty cache
    (3, 50, 60, 12, 3, 30),  # window longer than what was seen
])
def test_chunk_prefill_equals_prefill_rows_of_the_whole_sequence(S, W, ring_cap, Tc, n_sink, n_before):
    """With token values the codec stores exactly, prefilling a chunk against
    the cache gives exactly rows p0.. of the prefill of the whole sequence
    under make_causal_packing_mask (one segment, its first n_sink tokens
    sinks, the window): what the ring dropped is outside every chunk row's
    window, and the sinks are kept."""
    rng = philox(500 + S + W + Tc)
    B, Hq, Hkv, d = 2, 4, 2, 64
    T = n_sink + n_before + Tc
    k = _exact_int8_tokens(rng, (B, T, Hkv, d))
    v = _exact_int8_tokens(rng, (B, T, Hkv, d))
    q = rng.standard_normal((B, T, Hq, d))
    cache = oracle.Cache(B, Hkv, d, S, ring_cap)
    for t in range(n_sink + n_before):
        oracle.kv_append(cache, k[:, t], v[:, t], t < n_sink)
    p0 = n_sink + n_before
    out, lse, after = oracle.chunk_prefill(q[:, p0:], k[:, p0:], v[:, p0:], cache, W)
    seg = np.ones((B, T), np.int32)
    sink = np.zeros((B, T), np.uint8)
    sink[:, :n_sink] = 1
    want, wlse = oracle.swa_sink_prefill(q, k, v, seg, sink, W)
    np.testing.assert_allclose(out, want[:, p0:], atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, wlse[:, p0:], atol=1e-12, rtol=0)
    # the cache after the chunk is the cache after appending it token by token
    ref = cache.copy()
    for t in range(p0, T):
        oracle.kv_append(ref, k[:, t], v[:, t], False)
    for f in ("k_codes", "v_codes", "k_scale", "v_scale", "sink_len", "ring_start", "ring_len", "seq_len"):
        np.testing.assert_array_equal(getattr(after, f), getattr(ref, f))


def test_chunk_of_one_token_is_the_decode_of_that_token():
    """A one-token chunk is the decode step with the token's exact key: with
    codec-exact values, the chunk's output equals decode() after appending it."""
    rng = philox(510)
    B, Hq, Hkv, d, S, W = 3, 8, 2, 64, 4, 8
    cache = oracle.Cache(B, Hkv, d, S, W)
    k = _exact_int8_tokens(rng, (B, 20, Hkv, d))
    v = _exact_int8_tokens(rng, (B, 20, Hkv, d))
    for t in range(19):
        oracle.kv_append(cache, k[:, t], v[:, t], t < 3)
    q = rng.standard_normal((B, 1, Hq, d))
    out, _, after = oracle.chunk_prefill(q, k[:, 19:], v[:, 19:], cache, W)
    want, _ = oracle.decode(q[:, 0], after, W)
    np.testing.assert_allclose(out[:, 0], want, atol=1e-12, rtol=0)
