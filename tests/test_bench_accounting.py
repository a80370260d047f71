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


def test_fill_kept_tokens_matches_the_append_rule():
    """The handoff row's algorithmic bytes count the tokens the append rule
    keeps: the accepted sink prefix and the newest ring tokens."""
    seg = np.array([[1] * 10 + [2] * 6 + [0] * 2 + [3] * 5], np.int32)
    sink = np.zeros_like(seg, dtype=np.uint8)
    sink[0, :4] = 1          # segment 1: 4 sinks, 6 ring tokens
    sink[0, 10:16] = 1       # segment 2: sinks only
    kept, n = bench.fill_kept_tokens(seg, sink, S=3, W=4)
    assert n == 3
    assert kept == (3 + 4) + (3 + 0) + (0 + 4)


def test_rows_cover_every_measured_configuration():
    assert set(bench.ALL_ROWS) >= {"step_b64", "sweep", "packed", "compressed", "compressed_b8", "tiny", "pool",
                                   "append", "fill", "cdecode", "wsweep"}
    r = bench.roofline("hbm", 6e9, 1.0, 6000.0, "GB/s", "k", "measured")
    assert abs(r["achieved"] - 6000.0) < 1e-9 and abs(r["frac"] - 1.0) < 1e-12


def test_visible_pairs_pinned_matches_the_oracle_mask():
    """The pinned compressed row's visible pairs equal the oracle's: with
    q = 0 every visible column scores 0, so each row's lse is the log of its
    visible column count."""
    import oracle
    rng = philox(78)
    for T, W, b, P in ((64, 8, 4, 5), (100, 17, 3, 0), (53, 6, 2, 53), (300, 40, 8, 100)):
        q = np.zeros((1, T, 1, 32))
        k, v = (rng.standard_normal((1, T, 1, 32)) for _ in range(2))
        _, lse = oracle.compressed_prefill_pinned(q, k, v, W, b, P, 0.0)
        n = int(np.rint(np.exp(lse)).sum())
        assert bench.visible_pairs_pinned(T, W, b, P) == n
