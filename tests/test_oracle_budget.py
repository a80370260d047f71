"""Pins for the oracle's KV budget window (CPU only).

kv_budget_window and effective_kv_window follow "How the 256-Token Sliding
Window Works with Tools as KV Sinks in Needle", section "Effective KV Window:
Bounding the Cache Size"; the constants follow
"256-token滑动窗口+KV sink：Needle 2工具钉住机制源码分析", section
"256 这个窗口宽度从哪来：内存预算计算器".  Pinned by hand-derived cases and by
maximality: the window is the largest multiple of 32 whose cache fits the
budget, unless a clamp applies.
"""
import numpy as np
import pytest

import oracle
from conftest import golden_path
from workloads import philox

BUDGET = 11 * 1024 * 1024 + 512 * 1024


def cases():
    for line in open(golden_path("budget_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        lhs, rhs = line.split("|")
        yield [int(x) for x in lhs.split()], [int(x) for x in rhs.split()]


@pytest.mark.parametrize("args,want", list(cases()))
def test_hand_cases(args, want):
    d, a, h, kvh, L, sites, mx, kvw = args
    got = oracle.kv_budget_window(d, a, h, kvh, L, sites, mx)
    assert got == want[0]
    assert oracle.effective_kv_window(got, kvw) == want[1]


def test_budget_constant():
    assert BUDGET == 12058624


def cache_bytes_per_position(d, a, h, kvh, L, sites):
    """Bytes a position costs, counted item by item: per layer K and V codes
    (one byte per channel) and K and V scales (4 bytes per 32 channels); per
    engram site d_model bytes plus one 32-entry fp32 row."""
    hd = (a or d) // h
    channels = kvh * hd
    per_layer = 0
    for _tensor in ("K", "V"):
        per_layer += channels            # int8 codes
        per_layer += (channels // 32) * 4  # fp32 scales
    return L * per_layer + sites * (d + 32 * 4)


def test_window_is_largest_fitting_multiple_of_32():
    rng = philox(61)
    for _ in range(300):
        h = int(rng.choice([1, 2, 4, 8, 16]))
        kvh = int(rng.choice([1, 2, 4])) if h >= 4 else 1
        d = int(rng.choice([64, 128, 256, 512, 1024, 2048]))
        L = int(rng.integers(1, 40))
        sites = int(rng.integers(0, 4))
        mx = int(rng.integers(1, 70000))
        got = oracle.kv_budget_window(d, 0, h, kvh, L, sites, mx)
        pp = cache_bytes_per_position(d, 0, h, kvh, L, sites)
        fit = None
        w = 0
        while (w + 32) * pp <= BUDGET:     # largest multiple of 32 that fits
            w += 32
        fit = w
        if got == 160 and min(fit, mx) <= 160:
            continue                        # floor applied
        assert got == min(fit, mx)
        assert got >= 160
