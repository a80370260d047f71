"""GPU parity: chunked prefill against the bounded int8 cache
(nd_swa_sink_chunk_prefill) -- each new token of the chunk attends, under the
decode mask ("256-token 滑动窗口：源码走读": causal, sink at any distance or
within the window), to the cached sinks and ring entries and to the chunk's
own keys; then the chunk is ring-appended to the cache.  Outputs and lse
against oracle.chunk_prefill within the bf16 tolerance; the cache afterwards
bit for bit against the oracle's appends."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev, dev_bf16, host, need_gpu, no_device_errors
from workloads import decode_cache, normal_bf16, philox, random_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    no_device_errors()


def nd():
    import sliding_window_kv_swa_gb300 as m
    return m


def caches(w, S, W):
    B, Hkv, _, d = w["k"].shape
    ref = oracle.Cache(B, Hkv, d, S, W)
    ref.k_codes[...], ref.k_scale[...] = oracle.quant_g32(w["k"])
    ref.v_codes[...], ref.v_scale[...] = oracle.quant_g32(w["v"])
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        getattr(ref, f)[...] = w[f]
    gpu = nd().KVCache(*(dev(getattr(ref, f)) for f in ("k_codes", "v_codes", "k_scale", "v_scale", "sink_len",
                                                      "ring_start", "ring_len", "seq_len")), S, W)
    return ref, gpu


def check_cache(gpu, ref):
    for f in ("k_codes", "v_codes", "k_scale", "v_scale", "sink_len", "ring_start", "ring_len", "seq_len"):
        np.testing.assert_array_equal(host(getattr(gpu, f)), getattr(ref, f), err_msg=f)


def run_chunk(gpu, qb, kb, vb, window):
    B, Tc, Hq, d = qb.shape
    lse = torch.empty((B, Hq, Tc), dtype=torch.float32, device="cuda")
    out = nd().nd_swa_sink_chunk_prefill(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), gpu, window, lse=lse)
    return host(out), host(lse).transpose(0, 2, 1)


@pytest.mark.parametrize("Hq,Hkv,d,S,ring_cap,W,Tc,full", [
    (8, 2, 64, 24, 40, 40, 37, True),      # wrapped ring, GQA pairs
    (6, 2, 128, 16, 48, 20, 300, False),   # partial rings, window < ring, 3 heads per KV head
    (4, 4, 64, 8, 16, 16, 1, True),        # a one-token chunk
    (16, 8, 128, 0, 64, 64, 130, True),    # no sink slots
])
def test_chunk_prefill_matches_oracle(Hq, Hkv, d, S, ring_cap, W, Tc, full):
    rng = philox(5000 + Hq + d + Tc)
    B = 5
    w = decode_cache(B, Hq, Hkv, d, S, ring_cap, seed=5001 + Tc, full=full)
    ref, gpu = caches(w, S, ring_cap)
    if not full:
        ref.sink_len[:] = np.minimum(np.arange(B) * 5, S)
        ref.seq_len[:] = ref.sink_len + ref.ring_len
        gpu.sink_len.copy_(torch.from_numpy(ref.sink_len))
        gpu.seq_len.copy_(torch.from_numpy(ref.seq_len))
    qb, q = normal_bf16(rng, (B, Tc, Hq, d))
    kb, k = normal_bf16(rng, (B, Tc, Hkv, d))
    vb, v = normal_bf16(rng, (B, Tc, Hkv, d))
    got, glse = run_chunk(gpu, qb, kb, vb, W)
    want, wlse, after = oracle.chunk_prefill(q, k, v, ref, W)
    assert_close_bf16(got, want, "chunk prefill")
    np.testing.assert_allclose(glse, wlse, atol=2e-2, rtol=0)
    check_cache(gpu, after)


def test_two_chunks_then_a_decode_step():
    """Continuation: chunk, chunk, decode step -- each against the oracle
    sequence, the cache carried by the library between the calls."""
    rng = philox(5100)
    B, Hq, Hkv, d, S, W = 3, 8, 2, 128, 32, 64
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=5101, full=True)
    ref, gpu = caches(w, S, W)
    for Tc in (100, 45):
        qb, q = normal_bf16(rng, (B, Tc, Hq, d))
        kb, k = normal_bf16(rng, (B, Tc, Hkv, d))
        vb, v = normal_bf16(rng, (B, Tc, Hkv, d))
        got, _ = run_chunk(gpu, qb, kb, vb, W)
        want, _, ref = oracle.chunk_prefill(q, k, v, ref, W)
        assert_close_bf16(got, want, f"chunk of {Tc}")
    check_cache(gpu, ref)
    kb, kf = normal_bf16(rng, (B, Hkv, d))
    vb, vf = normal_bf16(rng, (B, Hkv, d))
    qb, qf = normal_bf16(rng, (B, Hq, d))
    out = nd().nd_swa_sink_decode_step(dev_bf16(qb), gpu, dev_bf16(kb), dev_bf16(vb), W)
    oracle.kv_append(ref, kf, vf, False)
    want, _ = oracle.decode(qf, ref, W)
    assert_close_bf16(host(out), want, "decode after the chunks")


def test_chunk_prefill_full_size():
    """A 4096-token chunk (the chunk size of long-prompt continuation) per
    sequence against the large-batch cache layout (Hq32 Hkv8 d128, 1024 sinks
    + a full 256-slot ring, W256), B4: every row and head against the
    oracle; the cache after the chunk bit for bit."""
    rng = philox(5200)
    B, Hq, Hkv, d, S, W, Tc = 4, 32, 8, 128, 1024, 256, 4096
    kc, ks, vc, vs = random_codes(rng, B, Hkv, S + W, d)
    ring_start = rng.integers(0, W, size=B).astype(np.int32)
    ref = oracle.Cache(B, Hkv, d, S, W)
    ref.k_codes[...], ref.k_scale[...], ref.v_codes[...], ref.v_scale[...] = kc, ks, vc, vs
    ref.sink_len[:] = S
    ref.ring_len[:] = W
    ref.ring_start[:] = ring_start
    ref.seq_len[:] = S + W + ring_start
    gpu = nd().KVCache(*(dev(getattr(ref, f)) for f in ("k_codes", "v_codes", "k_scale", "v_scale", "sink_len",
                                                      "ring_start", "ring_len", "seq_len")), S, W)
    qb, q = normal_bf16(rng, (B, Tc, Hq, d))
    kb, k = normal_bf16(rng, (B, Tc, Hkv, d))
    vb, v = normal_bf16(rng, (B, Tc, Hkv, d))
    got, glse = run_chunk(gpu, qb, kb, vb, W)
    want, wlse, after = oracle.chunk_prefill(q, k, v, ref, W)
    assert_close_bf16(got, want, "4096-token chunk")
    for b in range(B):
        assert_close_bf16(got[b], want[b], f"sequence {b}")
    np.testing.assert_allclose(glse, wlse, atol=2e-2, rtol=0)
    check_cache(gpu, after)
