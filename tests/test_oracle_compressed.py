"""Pins for the oracle's compressed-attention pieces (CPU only).

Follows "Compressed attention and the copy probe": compressed_mask (section
"Two kinds of columns, pooled blocks and exact recent keys") and _compress
(section "Pool before rotating, not after").  Pins: the page's invariants (no
token counted twice, early rows see only exact keys, blocks arrive one at a
time), its printed cache figure (4 MiB -> about 1.2 MiB), closed-form column
counts, the block-1 reduction to plain causal attention, numpy's mean, and the
geometry of the rotation (angles, norms, relative positions).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_path
from workloads import philox


def read_kv(name):
    out = {}
    for line in open(golden_path(name)):
        if line.strip() and not line.startswith("#"):
            k, v = line.split(":")
            out[k.strip()] = float(v)
    return out


def test_printed_cache_reduction():
    g = read_kv("compressed_cache.txt")
    T, W, b = int(g["T"]), int(g["window"]), int(g["block"])
    m = oracle.compressed_mask(T, W, b)
    kept = int(m[T - 1].sum())             # columns the last row keeps
    assert kept == (T - W) // b + W == 1216
    mib = g["full_mib"] * kept / T
    assert abs(mib - g["printed_mib"]) <= g["printed_precision_mib"]


def test_column_counts_closed_form():
    # exact: sum_q min(q+1, 256) = 256*257/2 + 3840*256;
    # pooled: sum_q floor((q-255)/4) over q >= 259 = 4*(959*960/2) + 960.
    m = oracle.compressed_mask(4096, 256, 4)
    nb = 1024
    assert int(m[:, nb:].sum()) == 32896 + 983040 == 1015936
    assert int(m[:, :nb].sum()) == 1841280 + 960 == 1842240


@pytest.mark.parametrize("T,W,b", [(64, 8, 4), (61, 5, 3), (40, 16, 8), (33, 1, 2)])
def test_no_token_counted_twice_and_blocks_arrive_in_order(T, W, b):
    m = oracle.compressed_mask(T, W, b)
    nb = T // b
    prev = 0
    for q in range(T):
        covered = []
        for j in np.nonzero(m[q, :nb])[0]:
            covered.extend(range(j * b, j * b + b))
        exact = list(np.nonzero(m[q, nb:])[0])
        assert len(set(covered)) == len(covered)
        assert not set(covered) & set(exact)                      # disjoint
        assert all(p <= q for p in covered + exact)               # causal
        n = int(m[q, :nb].sum())
        if q < W + b - 1:
            assert n == 0                                         # exact keys only
        assert prev <= n <= prev + 1                              # one block at a time
        # once a block clears the window its columns stay visible
        assert list(np.nonzero(m[q, :nb])[0]) == list(range(n))
        prev = n
        # every position is reached, either exactly or through its block,
        # except positions in a block that has not fully left the window
        if q >= W:
            assert set(covered) | set(exact) == set(range(len(covered))) | set(exact)


def test_pool_is_numpy_block_mean():
    rng = philox(51)
    x = rng.standard_normal((2, 23, 3, 8))
    for b in (1, 2, 4, 5):
        nb = 23 // b
        want = x[:, :nb * b].reshape(2, nb, b, 3, 8).mean(axis=2)
        np.testing.assert_allclose(oracle.pool_blocks(x, b), want, atol=1e-15, rtol=0)


def test_pool_constant_block_is_constant():
    x = np.repeat(np.arange(6.0)[None, :, None, None], 4, axis=1).reshape(1, 24, 1, 1)
    x = np.broadcast_to(x, (1, 24, 1, 4)).copy()
    np.testing.assert_array_equal(oracle.pool_blocks(x, 4)[0, :, 0, 0], np.arange(6.0))


def test_rope_geometry():
    rng = philox(52)
    d, theta = 16, 10000.0
    x = rng.standard_normal((1, 5, 2, d))
    pos = np.array([0, 1, 7, 100, 4095])
    r = oracle.rope(x, pos, theta)
    np.testing.assert_array_equal(r[0, 0], x[0, 0])                  # position 0: identity
    half = d // 2
    for i in range(half):                                          # each pair keeps its norm
        np.testing.assert_allclose(np.hypot(r[..., i], r[..., i + half]),
                                   np.hypot(x[..., i], x[..., i + half]), rtol=1e-13)
    # pair 0 turns by m radians (theta^0 = 1), counter-clockwise from (x_0, x_{d/2})
    for t, m in enumerate(pos):
        a0 = math.atan2(x[0, t, 0, half], x[0, t, 0, 0])
        a1 = math.atan2(r[0, t, 0, half], r[0, t, 0, 0])
        assert abs(math.remainder(a1 - a0 - m, 2 * math.pi)) < 1e-9
    # the last pair turns by m * theta^(-(d-2)/d)
    f = theta ** (-(d - 2) / d)
    a0 = math.atan2(x[0, 3, 1, d - 1], x[0, 3, 1, half - 1])
    a1 = math.atan2(r[0, 3, 1, d - 1], r[0, 3, 1, half - 1])
    assert abs(math.remainder(a1 - a0 - 100 * f, 2 * math.pi)) < 1e-9


def test_rope_scores_depend_on_offset_only():
    rng = philox(53)
    d = 32
    q = rng.standard_normal((1, 1, 1, d))
    k = rng.standard_normal((1, 1, 1, d))
    ref = None
    for m, n in [(5, 2), (103, 100), (4000, 3997)]:
        s = float((oracle.rope(q, np.array([m]), 1e4) * oracle.rope(k, np.array([n]), 1e4)).sum())
        ref = s if ref is None else ref
        assert abs(s - ref) < 1e-9


def test_pooled_key_rotated_at_block_midpoint():
    # d = 2: the rotation angle of pair 0 equals the position, so the angle of
    # each pooled key reveals the position it was rotated at.
    B, T, H, d = 1, 24, 1, 2
    for b in (1, 2, 3, 4, 8):
        k = np.zeros((B, T, H, d))
        k[..., 0] = 1.0                                            # angle 0 before rotation
        q = np.zeros_like(k)
        v = np.zeros_like(k)
        _, kk, _ = oracle.compress(q, k, v, b, theta=10.0)
        for j in range(T // b):
            ang = math.atan2(kk[0, j, 0, 1], kk[0, j, 0, 0])
            mid = j * b + b // 2
            assert abs(math.remainder(ang - mid, 2 * math.pi)) < 1e-9, (b, j)
        # exact keys follow, rotated at their own positions
        for t in range(T):
            ang = math.atan2(kk[0, T // b + t, 0, 1], kk[0, T // b + t, 0, 0])
            assert abs(math.remainder(ang - t, 2 * math.pi)) < 1e-9


@pytest.mark.parametrize("b,table_len", [(4, 10), (3, 7), (8, 1), (2, 24)])
def test_pooled_midpoint_clamped_to_rotary_table(b, table_len):
    # [C3] "Pool before rotating, not after" clamps each block midpoint to the
    # last row of the rotary table.  With a table shorter than T, blocks whose
    # midpoint j*b + b//2 lies past it are rotated at table_len - 1 instead;
    # d = 2 again, so the angle read back is the position used.
    B, T, H, d = 1, 24, 1, 2
    k = np.zeros((B, T, H, d))
    k[..., 0] = 1.0
    z = np.zeros_like(k)
    _, kk, _ = oracle.compress(z, k, z, b, theta=10.0, table_len=table_len)
    clamped = 0
    for j in range(T // b):
        mid = j * b + b // 2
        want = mid if mid <= table_len - 1 else table_len - 1
        clamped += want != mid
        ang = math.atan2(kk[0, j, 0, 1], kk[0, j, 0, 0])
        assert abs(math.remainder(ang - want, 2 * math.pi)) < 1e-9, (b, j, want)
    assert clamped == sum(1 for j in range(T // b) if j * b + b // 2 > table_len - 1)


def test_pool_happens_before_rotation():
    # Two keys of opposite angle offsets around the midpoint would shrink if
    # rotated first; pooling first keeps the mean of the raw keys, rotated once.
    B, T, H, d = 1, 8, 1, 4
    rng = philox(54)
    k = rng.standard_normal((B, T, H, d))
    _, kk, _ = oracle.compress(np.zeros_like(k), k, np.zeros_like(k), 4, theta=100.0)
    pooled = oracle.pool_blocks(k, 4)
    want = oracle.rope(pooled, np.array([2, 6]), 100.0)
    np.testing.assert_allclose(kk[:, :2], want, atol=1e-14, rtol=0)


@pytest.mark.parametrize("theta", [0.0, 10000.0])
def test_block_one_reduces_to_full_causal(theta):
    # b = 1: pooled column j is token j rotated at j, visible once it leaves the
    # window; together with the exact window that is every causal key once.
    rng = philox(55)
    B, T, H, d, W = 2, 40, 3, 8, 6
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    out, _ = oracle.compressed_prefill(q, k, v, W, 1, theta)
    if theta:
        pos = np.arange(T)
        q, k = oracle.rope(q, pos, theta), oracle.rope(k, pos, theta)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(out, want.permute(0, 2, 1, 3).numpy(), atol=1e-12, rtol=0)


def test_compressed_attention_matches_sdpa_on_concatenated_columns():
    rng = philox(56)
    B, T, H, d, W, b = 1, 48, 2, 8, 8, 4
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    out, _ = oracle.compressed_prefill(q, k, v, W, b, 1e4)
    qr, kk, vv = oracle.compress(q, k, v, b, 1e4)
    m = torch.from_numpy(oracle.compressed_mask(T, W, b))
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (qr, kk, vv))
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m)
    np.testing.assert_allclose(out, want.permute(0, 2, 1, 3).numpy(), atol=1e-12, rtol=0)


# ---------------------------------------------------------------- compressed decode cache
# The oracle's compressed-attention decode (compressed_cache / compressed_decode)
# stores every key and value as int8 group-32 codes; these pins tie it to the
# dense definition above.  Tolerance: int8 quantisation moves each stored
# element by at most scale/2 = amax/254 (about 1e-2 for N(0,1) groups), plus one
# bf16 rounding; the attention output of these small cases stays within 3e-2
# max / 6e-3 mean of the unquantised result, while one pooled column too many
# or too few (a visibility rule off by one) moves it by ~1/(columns) ~ 1e-1.
QMAX, QMEAN = 3e-2, 6e-3


@pytest.mark.parametrize("T,W,b", [(48, 8, 4), (40, 4, 4), (37, 5, 3), (30, 6, 1)])
def test_compressed_cache_columns_follow_the_mask(T, W, b):
    """At every query position the cache holds exactly the columns of that
    row of compressed_mask: the visible pooled blocks (sink_len) and the
    exact keys (ring positions)."""
    rng = philox(60 + T)
    k, v = (rng.standard_normal((1, T, 2, 32)) for _ in range(2))
    m = oracle.compressed_mask(T, W, b)
    for pos in range(T):
        c = oracle.compressed_cache(k, v, pos, W, b, 1e4, sink_cap=T // b + 1)
        assert int(c.sink_len[0]) == int(m[pos, :T // b].sum()), pos
        kpos, _ = oracle.slot_positions(c, 0)
        ring = sorted(int(x) for x in kpos[c.sink_cap:] if x >= 0)
        assert ring == [int(t) for t in np.nonzero(m[pos, T // b:])[0]], pos


@pytest.mark.parametrize("T,W,b", [(48, 8, 4), (40, 4, 4), (37, 5, 3)])
def test_compressed_decode_matches_compressed_prefill_rows(T, W, b):
    """Decode at every position equals the row of the dense compressed
    attention, up to the int8 storage."""
    rng = philox(70 + T)
    B, H, d = 2, 2, 64
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    want, _ = oracle.compressed_prefill(q, k, v, W, b, 1e4)
    errs = []
    for pos in range(T):
        out, _, _ = oracle.compressed_decode(q[:, pos], k, v, pos, W, b, 1e4)
        errs.append(np.abs(out - want[:, pos]))
    errs = np.stack(errs)
    assert errs.max() <= QMAX and errs.mean() <= QMEAN, (errs.max(), errs.mean())


def test_compressed_decode_with_pinned_prefix_block_one_is_causal_attention():
    """Pinned prefix + compressed attention with block 1: every token is kept
    (pinned, pooled singly at its own position, or in the window), so the
    decode equals plain causal attention up to the int8 storage; and a
    window as long as the sequence never pools."""
    rng = philox(80)
    B, T, H, d, P, W = 1, 30, 2, 32, 5, 4
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    pos_all = np.arange(T)
    qr, kr = oracle.rope(q, pos_all, 1e4), oracle.rope(k, pos_all, 1e4)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (qr, kr, v))
    full = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True).permute(0, 2, 1, 3).numpy()
    for pos in range(T):
        out, _, c = oracle.compressed_decode(q[:, pos], k, v, pos, W, 1, 1e4, n_pinned=P, sink_cap=T)
        assert np.abs(out - full[:, pos]).max() <= QMAX, pos
        assert int(c.sink_len[0]) == min(pos + 1, P) + max(0, pos - W + 1 - P)
    out, _, c = oracle.compressed_decode(q[:, T - 1], k, v, T - 1, T, 4, 1e4, n_pinned=P, ring_cap=T)
    assert int(c.sink_len[0]) == P and int(c.ring_len[0]) == T - P
    assert np.abs(out - full[:, T - 1]).max() <= QMAX


def test_pinned_tokens_are_seen_at_any_distance():
    """A pinned token's value reaches a query far past the window; the same
    token unpinned reaches it only through its block's mean (a quarter of
    the weight at block 4), and not at all before its block is visible."""
    rng = philox(81)
    B, T, H, d, W, b = 1, 64, 1, 32, 8, 4
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    v2 = v.copy()
    v2[:, 0] += 10.0
    pos = T - 1
    for P in (1, 0):
        a, _, _ = oracle.compressed_decode(q[:, pos], k, v, pos, W, b, 1e4, n_pinned=P)
        c_, _, _ = oracle.compressed_decode(q[:, pos], k, v2, pos, W, b, 1e4, n_pinned=P)
        assert np.abs(c_ - a).max() > 1e-2, P
    # token 0 unpinned, query at pos W + 1: block 0 (tokens 0..3) not yet visible
    a, _, _ = oracle.compressed_decode(q[:, W + 1], k, v, W + 1, W, b, 1e4)
    c_, _, _ = oracle.compressed_decode(q[:, W + 1], k, v2, W + 1, W, b, 1e4)
    np.testing.assert_array_equal(a, c_)


# ---------------------------------------------------------------- pinned prefix + compressed prefill

@pytest.mark.parametrize("theta", [0.0, 10000.0])
def test_pinned_compressed_prefill_without_pins_is_the_compressed_prefill(theta):
    rng = philox(90)
    B, T, H, d, W, b = 2, 53, 2, 16, 7, 4
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    got, gl = oracle.compressed_prefill_pinned(q, k, v, W, b, 0, theta)
    want, wl = oracle.compressed_prefill(q, k, v, W, b, theta)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)
    np.testing.assert_allclose(gl, wl, atol=1e-12, rtol=0)


@pytest.mark.parametrize("P", [1, 6, 40])
def test_pinned_compressed_prefill_block_one_is_causal_attention(P):
    """Block 1: pinned keys, single-token blocks at their own positions and the
    window cover every causal key once -- plain causal attention (SDPA)."""
    rng = philox(91 + P)
    B, T, H, d, W = 1, 40, 2, 16, 5
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    got, _ = oracle.compressed_prefill_pinned(q, k, v, W, 1, P, 10000.0)
    pos = np.arange(T)
    qr, kr = oracle.rope(q, pos, 1e4), oracle.rope(k, pos, 1e4)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (qr, kr, v))
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)


@pytest.mark.parametrize("P", [0, 5])
def test_pinned_compressed_prefill_rows_match_the_compressed_decode(P):
    """Every row of the prefill equals the compressed decode at that position
    (the same reading of pinned + pooled + window) within the int8 storage
    error of the decode's cache."""
    rng = philox(95 + P)
    B, T, H, d, W, b = 2, 46, 2, 64, 6, 4
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    pre, _ = oracle.compressed_prefill_pinned(q, k, v, W, b, P, 1e4)
    errs = []
    for t in range(T):
        out, _, _ = oracle.compressed_decode(q[:, t], k, v, t, W, b, 1e4, n_pinned=P)
        errs.append(np.abs(out - pre[:, t]))
    errs = np.stack(errs)
    assert errs.max() <= QMAX and errs.mean() <= QMEAN, (errs.max(), errs.mean())
