"""GPU test of the bounded-wait failure path, without a GPU fault.

Every mbarrier wait of the tensor-core prefill is bounded; one that gives up
raises device flag 1, and the kernel stops issuing work, lets what is in
flight land, frees its tensor memory and returns.  Here the epilogue's wait
for a row block's last P*V -- a wait that guards no copy in flight -- is put
in test mode (nd_set_prefill_epilogue_wait_limit): it polls a barrier that
nothing arrives on, 64 times, so it runs out on every CTA.  The call must
return, the flag must be raised, and the next calls (prefill and decode) on
the same context must be exact again."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev, dev_bf16, host, need_gpu
from workloads import decode_b64, normal_bf16, packed_segments, philox

pytestmark = pytest.mark.gpu


def nd():
    import sliding_window_kv_swa_gb300 as m
    return m


@pytest.mark.parametrize("d,Hq,Hkv", [(64, 4, 2), (128, 3, 1)])
def test_prefill_wait_that_runs_out_raises_the_flag_and_the_context_stays_usable(d, Hq, Hkv):
    need_gpu()
    lib = nd()
    rng = philox(6000 + d)
    B, T, W = 2, 600, 128
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    seg, sink = packed_segments(rng, B, T, 2, 3, 150, 3, 40)
    args = (dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), dev(seg), dev(sink), W)
    want, _ = oracle.swa_sink_prefill(q, k, v, seg, sink, W, 10000.0)
    torch.cuda.synchronize()
    assert lib.nd_device_errors(clear=True) == 0
    assert_close_bf16(host(lib.nd_swa_sink_prefill(*args, rope_theta=10000.0)), want, "before")
    torch.cuda.synchronize()
    try:
        lib.nd_set_prefill_epilogue_wait_limit(64)
        lib.nd_swa_sink_prefill(*args, rope_theta=10000.0)   # returns; its output is undefined
        torch.cuda.synchronize()
        flags = lib.nd_device_errors(clear=True)
    finally:
        lib.nd_set_prefill_epilogue_wait_limit(0)
    assert flags & 1, f"the wait that ran out must raise flag 1 (got {flags})"
    # the context is intact: the same call is exact again, and other kernels run
    assert_close_bf16(host(lib.nd_swa_sink_prefill(*args, rope_theta=10000.0)), want, "after")
    w = decode_b64()
    ref = oracle.Cache(64, 2, 64, 64, 256)
    ref.k_codes[...], ref.k_scale[...] = oracle.quant_g32(w["k"])
    ref.v_codes[...], ref.v_scale[...] = oracle.quant_g32(w["v"])
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        getattr(ref, f)[...] = w[f]
    cache = lib.KVCache(*(dev(getattr(ref, f)) for f in ("k_codes", "v_codes", "k_scale", "v_scale", "sink_len",
                                                       "ring_start", "ring_len", "seq_len")), 64, 256)
    out = lib.nd_swa_sink_decode(dev_bf16(w["q_bits"]), cache, 256)
    dw, _ = oracle.decode(w["q"], ref, 256)
    assert_close_bf16(host(out), dw, "decode after")
    torch.cuda.synchronize()
    assert lib.nd_device_errors(clear=True) == 0
