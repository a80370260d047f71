"""The benchmark's algorithmic-work bookkeeping (visible pairs, bytes) agrees
with the oracle's masks and the cache layout, so reported TFLOP/s and GB/s
count exactly the work the method defines."""
import numpy as np

import bench
import oracle
from workloads import packed_prefill, packed_segments, philox


def test_visible_pairs_packed_matches_oracle_mask():
    rng = philox(1500)
    for W in (1, 7, 64, 256):
        seg, sink = packed_segments(rng, 3, 900, 2, 4, 150, 3, 100)
        want = oracle.causal_packing_mask(seg, sink, W).sum(axis=(1, 2))
        np.testing.assert_array_equal(bench.visible_pairs_packed(seg, sink, W), want)


def test_visible_pairs_compressed_matches_oracle_mask():
    for T, W, b in ((4096, 256, 4), (300, 16, 3), (64, 8, 1)):
        assert bench.visible_pairs_compressed(T, W, b) == int(oracle.compressed_mask(T, W, b).sum())
    assert bench.visible_pairs_compressed(4096, 256, 4) == 2858176


def test_packed_workload_pair_count_in_expected_range():
    w = packed_prefill()
    pairs = bench.visible_pairs_packed(w["seg_ids"], w["sink"], w["window"])
    assert pairs.shape == (8,)
    assert 1.0e6 < pairs.mean() < 2.5e6        # vs 8.39e6 for plain causal at T=4096


def test_decode_bytes():
    cache, qo, app = bench.decode_bytes(64, 8, 2, 64, 64, 256)
    assert cache == 5898240                   # 64 seq x 320 slots x 2 heads x (2*64 + 2*2*4)
    assert qo == 2 * 64 * 8 * 64 * 2
    cache5, _, _ = bench.decode_bytes(512, 32, 8, 128, 1024, 256)
    assert cache5 == 512 * 1280 * 2304


def test_performed_tile_counts_bound_the_visible_tiles():
    """The prefill tile count the bench reports sits between the tiles that
    hold a visible pair (brute force on the oracle's mask) and all causal
    tiles."""
    import bench
    import oracle
    rng = philox(77)
    B, T, W, span, bn = 2, 700, 100, 128, 64
    seg, sink = packed_segments(rng, B, T, 2, 4, 120, 3, 40)
    mask = oracle.causal_packing_mask(seg, sink, W)   # [B][T][T] bool
    visible, causal = 0, 0
    for b in range(B):
        for q0 in range(0, T, span):
            q1 = min(T, q0 + span)
            for k0 in range(0, q1, bn):
                causal += 1
                visible += bool(mask[b, q0:q1, k0:k0 + bn].any())
    got = bench.performed_tiles_packed(seg, sink, W, span, bn)
    assert visible <= got <= causal, (visible, got, causal)
    # one segment, no sinks, no window: every causal tile
    seg1 = np.ones((1, T), np.int32)
    assert bench.performed_tiles_packed(seg1, np.zeros((1, T), np.uint8), 0, span, bn) == \
        sum((min(T, q0 + span) - 1) // bn + 1 for q0 in range(0, T, span))
