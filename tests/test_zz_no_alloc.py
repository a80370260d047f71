"""nd_swa_sink_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a serving loop that must not call cudaMalloc, a host
runtime that owns all device memory).  Its split-K scratch is a fixed device
array inside the library; these tests call it through the C ABI and check it
against nd_swa_sink_decode with a caller workspace and against the oracle, on
two calls in a row (the second call reuses the scratch the first one left
behind), and check that shapes needing more scratch than the array holds, and
shapes the workspace entry point refuses, are refused with the same status.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev, dev_bf16, host, need_gpu
from workloads import decode_cache, normal_bf16, philox

pytestmark = pytest.mark.gpu


def _caches(nd, w, S, W):
    ref = oracle.Cache(*w["k"].shape[:2], w["k"].shape[3], S, W)
    ref.k_codes[...], ref.k_scale[...] = oracle.quant_g32(w["k"])
    ref.v_codes[...], ref.v_scale[...] = oracle.quant_g32(w["v"])
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        getattr(ref, f)[...] = w[f]
    return ref, nd.KVCache(dev(ref.k_codes), dev(ref.v_codes), dev(ref.k_scale), dev(ref.v_scale),
                           dev(ref.sink_len), dev(ref.ring_start), dev(ref.ring_len), dev(ref.seq_len), S, W)


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    need_gpu()
    import sliding_window_kv_swa_gb300 as nd
    S, W = 64, 1024
    # 8 sequences x 2 KV heads are too few to fill the GPU and 1088 slots are
    # more than one step per warp, so the decode splits each sequence's slots
    # and needs scratch for the partials
    w = decode_cache(8, 8, 2, 64, S, W, seed=2023, full=True)
    B, Hq, d = w["q"].shape
    ref, cache = _caches(nd, w, S, W)
    need = nd.nd_swa_sink_decode_workspace_size(B, Hq, cache.n_kv_heads, d, S + W)
    assert 0 < need <= nd.nd.NOALLOC_SCRATCH_BYTES
    rng = philox(2024)
    queries = [(w["q_bits"], w["q"]), normal_bf16(rng, (B, Hq, d))]
    for call, (q_bits, q_f32) in enumerate(queries):
        q = dev_bf16(q_bits)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        want = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        want_lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        nd.nd_swa_sink_decode(q, cache, W, out=want, lse=want_lse, workspace=ws)
        got = torch.empty_like(want)
        got_lse = torch.empty_like(want_lse)
        nd.nd_swa_sink_decode_noalloc(q, cache, W, out=got, lse=got_lse)
        torch.cuda.synchronize()
        assert_close_bf16(host(got), host(want), f"noalloc call {call}")
        np.testing.assert_allclose(host(got_lse), host(want_lse), atol=2e-3, rtol=0)
        ref_out, ref_lse = oracle.decode(q_f32, ref, W)
        assert_close_bf16(host(got), ref_out, f"noalloc call {call} vs oracle")
        np.testing.assert_allclose(host(got_lse), ref_lse, atol=2e-3, rtol=0)
    assert nd.nd_device_errors(clear=True) == 0


def test_noalloc_refuses_what_the_workspace_decode_refuses():
    """Shapes the workspace entry point refuses get the same status here,
    not ND_ERR_WORKSPACE, even when they are large."""
    need_gpu()
    import sliding_window_kv_swa_gb300 as nd
    B, Hkv, d, S, W = 2, 8, 128, 1024, 256
    cache = nd.KVCache.empty(B, Hkv, d, S, W)
    for Hq, want in ((80, nd.nd.ND_ERR_UNSUPPORTED),   # 10 query heads per KV head (at most 8)
                     (12, nd.nd.ND_ERR_INVALID_ARG)):  # not a multiple of the KV heads
        q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        out = torch.empty_like(q)
        for fn in (lambda: nd.nd_swa_sink_decode_noalloc(q, cache, W, out=out),
                   lambda: nd.nd_swa_sink_decode(q, cache, W, out=out,
                                                 workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))):
            with pytest.raises(nd.NDError) as ei:
                fn()
            assert ei.value.status == want


def test_noalloc_refuses_shapes_beyond_its_scratch():
    need_gpu()
    import sliding_window_kv_swa_gb300 as nd
    B, Hq, Hkv, d, S, W = 2, 64, 8, 128, 1024, 256   # ten-way split of 1280 slots
    need = nd.nd_swa_sink_decode_workspace_size(B, Hq, Hkv, d, S + W)
    assert need > nd.nd.NOALLOC_SCRATCH_BYTES
    cache = nd.KVCache.empty(B, Hkv, d, S, W)
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(nd.NDError) as ei:
        nd.nd_swa_sink_decode_noalloc(q, cache, W, out=out)
    assert ei.value.status == nd.nd.ND_ERR_WORKSPACE
