"""CPU checks of the C ABI: the library builds, loads, exports every entry point
nd.h declares, rejects bad arguments on the host, and its host-only budget
window equals the oracle's bit for bit.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import oracle
from conftest import ROOT
from workloads import philox


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "nd.h")).read()
    return sorted(set(re.findall(r"ND_API\s+[\w\s\*]*?\b(nd_\w+)\s*\(", src)))


def test_library_exports_every_declared_entry_point():
    import sliding_window_kv_swa_gb300 as nd
    lib = ctypes.CDLL(nd.library_path())
    names = declared_entry_points()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(nd.EXPORTED)


def test_version_and_status_strings():
    import sliding_window_kv_swa_gb300 as nd
    assert "sm_103a" in nd.nd_version()
    assert nd.nd_status_string(0) == "ND_OK"
    assert nd.nd_status_string(1) == "ND_ERR_INVALID_ARG"


def test_budget_window_matches_oracle():
    import sliding_window_kv_swa_gb300 as nd
    rng = philox(71)
    for _ in range(500):
        h = int(rng.choice([1, 2, 4, 8, 16, 32]))
        kvh = int(rng.choice([x for x in (1, 2, 4, 8) if x <= h]))
        d = int(rng.choice([64, 128, 256, 512, 1024, 4096]))
        a = int(rng.choice([0, 0, 256, 512]))
        L = int(rng.integers(0, 48))
        sites = int(rng.integers(0, 3))
        mx = int(rng.integers(1, 70000))
        kvw = int(rng.choice([0, 128, 256, 4096]))
        want = oracle.kv_budget_window(d, a, h, kvh, L, sites, mx)
        if want < 0:
            with pytest.raises(nd.NDError):
                nd.nd_kv_budget_window(d, a, h, kvh, L, sites, mx, kvw)
            continue
        b, e = nd.nd_kv_budget_window(d, a, h, kvh, L, sites, mx, kvw)
        assert b == want
        assert e == oracle.effective_kv_window(want, kvw)


def test_budget_window_rejects_bad_config():
    import sliding_window_kv_swa_gb300 as nd
    with pytest.raises(nd.NDError) as ei:
        nd.nd_kv_budget_window(512, 0, 0, 2, 12, 2, 4096)
    assert ei.value.status == 1
    with pytest.raises(nd.NDError):
        nd.nd_kv_budget_window(512, 0, 8, 2, 0, 0, 4096)   # per_pos == 0


def test_host_validation_before_any_device_work():
    import sliding_window_kv_swa_gb300 as nd
    lib = ctypes.CDLL(nd.library_path())
    lib.nd_swa_sink_prefill.restype = ctypes.c_int
    P = ctypes.c_void_p
    # bad dtype, head_dim, GQA ratio, negative window: all rejected on the host
    args = lambda dt, hq, hkv, d, w, blk=0, seg=None: (
        P(16), P(16), P(16), dt, 1, 8, hq, hkv, d, seg, None, w, ctypes.c_float(0.0),
        None, None, blk, P(16), None, None, ctypes.c_size_t(0), None)
    assert lib.nd_swa_sink_prefill(*args(7, 4, 1, 64, 0)) == 1
    assert lib.nd_swa_sink_prefill(*args(1, 4, 1, 96, 0)) == 2
    assert lib.nd_swa_sink_prefill(*args(1, 6, 4, 64, 0)) == 1
    assert lib.nd_swa_sink_prefill(*args(1, 4, 1, 64, -1)) == 1
    # compressed variant needs bf16, no segments, window >= 1, pooled tensors
    assert lib.nd_swa_sink_prefill(*args(0, 4, 1, 64, 8, blk=4)) == 2
    assert lib.nd_swa_sink_prefill(*args(1, 4, 1, 64, 0, blk=4)) == 1
    assert lib.nd_swa_sink_prefill(*args(1, 4, 1, 64, 8, blk=4, seg=P(16))) == 1
    # misaligned pointer
    bad = list(args(1, 4, 1, 64, 0))
    bad[0] = P(18)
    assert lib.nd_swa_sink_prefill(*bad) == 1
    # decode: window < 1 and G > 8
    cache = nd.nd._Cache(1, 1, 64, 4, 8, 16, 16, 16, 16, 16, 16, 16, 16)
    lib.nd_swa_sink_decode.restype = ctypes.c_int
    assert lib.nd_swa_sink_decode(P(16), ctypes.byref(cache), 1, 0, P(16), None, None,
                                  ctypes.c_size_t(0), None) == 1
    assert lib.nd_swa_sink_decode(P(16), ctypes.byref(cache), 16, 8, P(16), None, None,
                                  ctypes.c_size_t(0), None) == 2
    # workspace required when the decode splits (1 sequence, 64 + 1024 slots)
    big = nd.nd._Cache(1, 1, 64, 64, 1024, 16, 16, 16, 16, 16, 16, 16, 16)
    assert lib.nd_swa_sink_decode(P(16), ctypes.byref(big), 4, 256, P(16), None, None,
                                  ctypes.c_size_t(0), None) == 4
    # append: head_dim not a multiple of 32
    c2 = nd.nd._Cache(1, 1, 48, 4, 8, 16, 16, 16, 16, 16, 16, 16, 16)
    assert lib.nd_kv_append_quant(ctypes.byref(c2), P(16), P(16), 0, None) == 1
    # prefill -> cache handoff: a ring is required, the row map is required,
    # src_seg is required with seg_ids, k / v aligned, head_dim 32..256
    fill = lib.nd_kv_cache_from_prefill
    fill.restype = ctypes.c_int
    no_ring = nd.nd._Cache(1, 1, 64, 4, 0, 16, 16, 16, 16, 16, 16, 16, 16)
    W16, Z = P(16), ctypes.c_size_t
    assert fill(ctypes.byref(no_ring), P(16), P(16), 1, 8, None, None, P(16), None, W16, Z(1 << 20), None) == 1
    assert fill(ctypes.byref(cache), P(16), P(16), 1, 8, None, None, None, None, W16, Z(1 << 20), None) == 1
    assert fill(ctypes.byref(cache), P(16), P(16), 1, 8, P(16), None, P(16), None, W16, Z(1 << 20), None) == 1
    assert fill(ctypes.byref(cache), P(18), P(16), 1, 8, None, None, P(16), None, W16, Z(1 << 20), None) == 1
    assert fill(ctypes.byref(cache), P(16), P(16), -1, 8, None, None, P(16), None, W16, Z(1 << 20), None) == 1
    wide = nd.nd._Cache(1, 1, 512, 4, 8, 16, 16, 16, 16, 16, 16, 16, 16)
    assert fill(ctypes.byref(wide), P(16), P(16), 1, 8, None, None, P(16), None, W16, Z(1 << 20), None) == 2
    # the kept tokens' plan: one (position, slot) pair per slot and a count, per row
    need = nd.nd_kv_cache_from_prefill_workspace_size(1, 4, 8)
    assert need >= (1 + 2 * 12) * 4
    assert fill(ctypes.byref(cache), P(16), P(16), 1, 8, None, None, P(16), None, None, Z(need), None) == 4
    assert fill(ctypes.byref(cache), P(16), P(16), 1, 8, None, None, P(16), None, W16, Z(need - 16), None) == 4
    # pinned compressed prefill: block >= 1, window >= 1, 0 <= n_pinned <= T
    cp = lib.nd_compressed_prefill
    cp.restype = ctypes.c_int
    cargs = lambda win, blk, pin: (P(16), P(16), P(16), 1, 8, 4, 4, 64, win, blk, pin, ctypes.c_float(1e4), P(16),
                                   None, P(16), ctypes.c_size_t(1 << 20), None)
    assert cp(*cargs(8, 0, 0)) == 1
    assert cp(*cargs(0, 4, 0)) == 1
    assert cp(*cargs(8, 4, 9)) == 1
    assert cp(*cargs(8, 4, -1)) == 1
    # chunked prefill: window >= 1, a ring, GQA ratio, head_dim 64/128, workspace
    chunk = lib.nd_swa_sink_chunk_prefill
    chunk.restype = ctypes.c_int
    Z = ctypes.c_size_t
    call = lambda c, hq, win, ws, n: chunk(P(16), P(16), P(16), 8, ctypes.byref(c), hq, win, P(16), None, ws, Z(n),
                                           None)
    assert call(cache, 4, 0, P(16), 1 << 20) == 1
    assert call(no_ring, 4, 8, P(16), 1 << 20) == 1
    c3 = nd.nd._Cache(1, 3, 64, 4, 8, 16, 16, 16, 16, 16, 16, 16, 16)
    assert call(c3, 4, 8, P(16), 1 << 20) == 1
    c96 = nd.nd._Cache(1, 1, 96, 4, 8, 16, 16, 16, 16, 16, 16, 16, 16)
    assert call(c96, 4, 8, P(16), 1 << 20) == 2
    assert call(cache, 4, 8, None, 1 << 20) == 4
    assert call(cache, 4, 8, P(16), 16) == 4


def test_workspace_sizes():
    import sliding_window_kv_swa_gb300 as nd
    # one CTA per (sequence, KV head) once that fills half the GPU: no split
    assert nd.nd_swa_sink_decode_workspace_size(64, 8, 2, 64, 320) == 0
    assert nd.nd_swa_sink_decode_workspace_size(512, 32, 8, 128, 1280) == 0
    # 8 sequences x 2 KV heads, 320 slots: one 16-slot step for each of the
    # 20 warps already, no split; 1088 slots (68 steps): four-way split,
    # (64+2) floats per partial
    assert nd.nd_swa_sink_decode_workspace_size(8, 8, 2, 64, 320) == 0
    assert nd.nd_swa_sink_decode_workspace_size(8, 8, 2, 64, 1088) == 8 * 8 * 4 * 66 * 4
    # chunked prefill: gathered bf16 keys and values of sinks + window-1 ring
    # rows + the chunk, per sequence
    n = nd.nd_swa_sink_chunk_prefill_workspace_size(2, 100, 8, 2, 64, 16, 32, 8)
    assert n >= 2 * 2 * (16 + 7 + 100) * 2 * 64 * 2
    # prefill with rotation keeps rotated copies of q and k
    n = nd.nd_swa_sink_prefill_workspace_size(nd.ND_F32, 1, 512, 4, 1, 64, 10000.0, 0)
    assert n >= 512 * 4 * 64 * 4 + 512 * 1 * 64 * 4


def test_host_step_validation_before_any_device_work():
    """The host-buffer step forms reject missing buffers, a bad window and a
    missing or short workspace on the host, before touching a device."""
    import sliding_window_kv_swa_gb300 as nd
    lib = ctypes.CDLL(nd.library_path())
    P, Z = ctypes.c_void_p, ctypes.c_size_t
    for fn in ("nd_swa_sink_decode_step_host", "nd_swa_sink_decode_step_host_packed",
               "nd_swa_sink_decode_step_host_workspace_size"):
        getattr(lib, fn).restype = ctypes.c_size_t if fn.endswith("size") else ctypes.c_int
    lib.nd_swa_sink_decode_step_host_workspace_size.argtypes = [ctypes.c_int] * 5
    cache = nd.nd._Cache(2, 1, 64, 4, 8, 16, 16, 16, 16, 16, 16, 16, 16)
    need = lib.nd_swa_sink_decode_step_host_workspace_size(2, 4, 1, 64, 12)
    # q, k_new, v_new (128 x 2 B each ...) then out and lse, 16-byte multiples
    assert need >= 2 * 4 * 64 * 2 + 2 * (2 * 1 * 64 * 2) + 2 * 4 * 64 * 2
    packed = lambda inp, win, out, ws, n: lib.nd_swa_sink_decode_step_host_packed(
        inp, ctypes.byref(cache), 4, win, out, 1, ws, Z(n), None)
    assert packed(None, 8, P(16), P(16), need) == 1          # no input buffer
    assert packed(P(16), 8, None, P(16), need) == 1          # no output buffer
    assert packed(P(16), 0, P(16), P(16), need) == 1         # window < 1
    assert packed(P(16), 8, P(16), None, need) == 4          # no workspace
    assert packed(P(16), 8, P(16), P(16), need - 16) == 4    # short workspace
    assert packed(P(16), 8, P(16), P(24), need) == 4         # misaligned workspace
    sep = lambda q, k, v: lib.nd_swa_sink_decode_step_host(
        q, ctypes.byref(cache), k, v, 4, 8, P(16), None, P(16), Z(need), None)
    assert sep(P(16), None, P(16)) == 1
    assert sep(P(16), P(16), None) == 1
    assert sep(None, P(16), P(16)) == 1


def test_bf16_prefill_workspace_holds_no_rotated_q():
    """The bf16 prefill rotates q inside its attention kernel: with rotation
    its workspace adds only the rotated K and the angle table."""
    import sliding_window_kv_swa_gb300 as nd
    B, T, Hq, Hkv, d = 1, 512, 4, 1, 64
    with_rope = nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, Hq, Hkv, d, 10000.0, 0)
    no_rope = nd.nd_swa_sink_prefill_workspace_size(nd.ND_BF16, B, T, Hq, Hkv, d, 0.0, 0)
    k_bytes = B * T * Hkv * d * 2            # rotated K, bf16 (a multiple of 256 here)
    table_bytes = T * (d // 2) * 8           # (cos, sin) fp32 per position and pair
    assert with_rope - no_rope == k_bytes + table_bytes
    # the fp32 path still keeps rotated copies of both q and k; a problem this
    # small (at most 256 CTAs of 16 rows) splits its keys over four CTAs per
    # row tile, whose partial states -- D values, max and sum per row and
    # split -- follow
    f32 = nd.nd_swa_sink_prefill_workspace_size(nd.ND_F32, B, T, Hq, Hkv, d, 10000.0, 0)
    partials = B * Hq * T * 4 * (d + 2) * 4
    assert f32 == B * T * Hq * d * 4 + B * T * Hkv * d * 4 + table_bytes + partials
    # a large one does not split
    assert nd.nd_swa_sink_prefill_workspace_size(nd.ND_F32, 8, 4096, 32, 8, 128, 0.0, 0) == 0


def test_empty_problems_return_ok_without_a_device():
    """Every compute entry point returns ND_OK for an empty problem (no
    sequences, no tokens, no rows, no whole pooled block) before touching a
    device: on a machine without a GPU any device call would fail instead."""
    import sliding_window_kv_swa_gb300 as nd
    lib = ctypes.CDLL(nd.library_path())
    P, Z, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    empty = nd.nd._Cache(0, 2, 64, 4, 8, None, None, None, None, None, None, None, None)
    e = ctypes.byref(empty)
    calls = {
        "nd_kv_append_quant": (e, None, None, 0, None),
        "nd_kv_quant_rows": (None, ctypes.c_int64(0), 64, None, None, None),
        "nd_kv_cache_from_prefill": (e, None, None, 1, 16, None, None, None, None, None, Z(0), None),
        "nd_swa_sink_chunk_prefill": (None, None, None, 16, e, 4, 8, None, None, None, Z(0), None),
        "nd_compressed_prefill": (None, None, None, 0, 16, 4, 4, 64, 8, 4, 2, F(10000.0), None, None, None, Z(0),
                                  None),
        "nd_swa_sink_decode": (None, e, 4, 8, None, None, None, Z(0), None),
        "nd_swa_sink_decode_step": (None, e, None, None, 4, 8, None, None, None, Z(0), None),
        "nd_swa_sink_decode_step_host": (None, e, None, None, 4, 8, None, None, None, Z(0), None),
        "nd_swa_sink_decode_step_host_packed": (None, e, 4, 8, None, 0, None, Z(0), None),
        "nd_swa_sink_decode_noalloc": (None, e, 4, 8, None, None, None),
        "nd_swa_sink_prefill": (None, None, None, 1, 0, 16, 4, 2, 64, None, None, 0, F(10000.0),
                                None, None, 0, None, None, None, Z(0), None),
        "nd_rope_apply": (None, None, 0, 16, 2, 64, F(10000.0), None),
        "nd_kv_compress_pool": (None, None, 1, 3, 2, 64, 4, F(10000.0), None, None, None),
    }
    for fn, args in calls.items():
        f = getattr(lib, fn)
        f.restype = ctypes.c_int
        assert f(*args) == 0, fn
    # T = 0 with sequences present
    assert lib.nd_swa_sink_prefill(None, None, None, 1, 2, 0, 4, 2, 128, None, None, 0, F(0.0),
                                   None, None, 0, None, None, None, Z(0), None) == 0
