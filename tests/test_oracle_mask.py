"""Pins for the oracle's masks (CPU only).

The prefill mask follows make_causal_packing_mask ("How the 256-Token Sliding
Window Works with Tools as KV Sinks in Needle", section "KV Sinks for Tools");
the decode mask follows the three-line decode mask of
"256-token滑动窗口+KV sink：Needle 2工具钉住机制源码分析", section
"256-token 滑动窗口：源码走读".  Each pin checks the oracle against something
other than itself: an enumeration written per segment, closed-form pair
counts, the page's worked example, and invariants the pages state.
"""
import numpy as np
import pytest

import oracle
from conftest import golden_path
from workloads import philox, tiny_prefill


def visible_by_segment(seg, sink, window):
    """Independent enumeration: walk each segment's rows and list the keys a
    row may read -- its own segment's causal past, restricted to the last
    `window` positions, plus that segment's sink positions (any distance)."""
    T = len(seg)
    m = np.zeros((T, T), bool)
    t = 0
    while t < T:
        e = t
        while e < T and seg[e] == seg[t]:
            e += 1
        if seg[t] > 0:
            for q in range(t, e):
                lo = t if window == 0 else max(t, q - window + 1)
                for k in range(lo, q + 1):
                    m[q, k] = True
                if window != 0 and sink is not None:
                    for k in range(t, q + 1):
                        if sink[k]:
                            m[q, k] = True
        t = e
    return m


@pytest.mark.parametrize("seed", range(12))
def test_mask_matches_segment_enumeration(seed):
    rng = philox(100 + seed)
    T = int(rng.integers(1, 48))
    # contiguous segments (the packing the pages describe)
    n = int(rng.integers(1, 5))
    cuts = np.sort(rng.integers(0, T + 1, size=n - 1))
    seg = np.zeros(T, np.int32)
    bounds = np.concatenate(([0], cuts, [T]))
    for i in range(n):
        # packed runs carry distinct ids; some runs are padding (id 0)
        seg[bounds[i]:bounds[i + 1]] = 0 if rng.random() < 0.2 else i + 1
    sink = (rng.random(T) < 0.25).astype(np.uint8)
    window = int(rng.choice([0, 1, 2, 3, 5, 8, 64]))
    got = oracle.causal_packing_mask(seg[None], sink[None], window)[0]
    want = visible_by_segment(seg, sink, window)
    np.testing.assert_array_equal(got, want)


def test_needle_worked_example():
    rows = [l.split() for l in open(golden_path("needle_8x8_mask.txt")) if l.strip() and not l.startswith("#")]
    seg = np.array([int(x) for x in rows[0][1:]], np.int32)
    window = int(rows[1][1])
    want = np.array([[int(x) for x in r] for r in rows[2:]], bool)
    got = oracle.causal_packing_mask(seg[None], (seg == 1)[None], window)
    assert got.shape == (1, 8, 8)
    np.testing.assert_array_equal(got[0], want)


def test_pair_counts_tiny_prefill_literal():
    # seg 1 = 48 sink tokens, seg 2 = 464 tokens, W = 256:
    # seg 1 rows: 48*49/2 = 1176; seg 2 rows: 256*257/2 + 208*256 = 86144.
    w = tiny_prefill(single_segment=False)
    m = oracle.causal_packing_mask(w["seg_ids"], w["sink"], w["window"])
    assert int(m.sum()) == 87320


def test_pair_counts_tiny_prefill_single_segment():
    # rows 0..255: q+1; rows 256..302: 256 + (q-255); rows 303..511: 256 + 48.
    w = tiny_prefill(single_segment=True)
    m = oracle.causal_packing_mask(w["seg_ids"], w["sink"], w["window"])
    assert int(m.sum()) == 32896 + 13160 + 63536 == 109592


def test_window_zero_switches_window_off():
    # seg 1: 1176 pairs, seg 2: 464*465/2 = 107880.
    w = tiny_prefill(single_segment=False)
    m = oracle.causal_packing_mask(w["seg_ids"], w["sink"], 0)
    assert int(m.sum()) == 109056
    # with no window the sink flag changes nothing
    m2 = oracle.causal_packing_mask(w["seg_ids"], None, 0)
    np.testing.assert_array_equal(m, m2)


def test_wide_window_single_segment_is_causal():
    T = 512
    seg = np.ones((1, T), np.int32)
    m = oracle.causal_packing_mask(seg, None, T)
    assert int(m.sum()) == T * (T + 1) // 2 == 131328
    np.testing.assert_array_equal(m[0], np.tril(np.ones((T, T), bool)))


def test_sink_visible_at_any_distance_within_segment():
    w = tiny_prefill(single_segment=True)
    m = oracle.causal_packing_mask(w["seg_ids"], w["sink"], w["window"])[0]
    assert m[511, :48].all()            # distance up to 511 >> W
    assert not m[511, 100]              # a non-sink key outside the window
    assert m[511, 256:].all() and not m[511, 48:256].any()


def test_padding_rows_and_columns_masked():
    seg = np.array([[1, 1, 0, 0, 2, 2]], np.int32)
    m = oracle.causal_packing_mask(seg, np.ones_like(seg), 4)[0]
    assert not m[2].any() and not m[3].any()
    assert not m[:, 2].any() and not m[:, 3].any()


def test_decode_keep_brute_force():
    rng = philox(7)
    for _ in range(50):
        n = int(rng.integers(1, 40))
        kpos = rng.integers(0, 100, size=n)
        sink = rng.random(n) < 0.3
        qpos = int(rng.integers(0, 100))
        W = int(rng.integers(1, 50))
        got = oracle.decode_keep(qpos, kpos, sink, W)
        for i in range(n):
            inside = qpos - W < kpos[i] <= qpos
            assert got[i] == ((kpos[i] <= qpos) and (inside or bool(sink[i])))
