"""GPU parity: compressed-attention decode (nd_compressed_decode_step) against
the oracle ("Compressed attention and the copy probe": one softmax over the
visible pooled blocks and the exact window, pooled keys rotated at their block
midpoint; optionally a pinned sink prefix).

Sequences are decoded step by step from an empty cache.  Outputs (and lse)
are compared with oracle.compressed_decode at the same position within the
bf16 tolerance; the cache's metadata with the oracle's exactly; and its codes
bit for bit with what the library's own pooling, rotation and codec entry
points produce from the same tokens (the incremental pooler must write the
same blocks as the bulk one)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev, dev_bf16, host, need_gpu, no_device_errors
from workloads import compressed, normal_bf16, philox

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    no_device_errors()


def nd():
    import sliding_window_kv_swa_gb300 as m
    return m


def run_steps(qb, kb, vb, W, block, theta, n_pinned, ring_cap, check_at, Hq):
    """Decode positions 0..T-1 one step at a time; returns the cache and the
    outputs / lse at the positions in check_at."""
    B, T, Hkv, d = kb.shape
    n_blk = max(0, (T - n_pinned) // block)
    cache = nd().CompressedCache.empty(B, Hkv, d, n_blk, ring_cap, block, n_pinned)
    st = cache.struct()
    ws = torch.empty(nd().nd_compressed_decode_step_workspace_size(B, Hq, Hkv, d, n_pinned + n_blk + ring_cap),
                     dtype=torch.uint8, device="cuda")
    q_d, k_d, v_d = dev_bf16(qb), dev_bf16(kb), dev_bf16(vb)
    outs = {}
    for p in range(T):
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        nd().nd_compressed_decode_step(q_d[:, p].contiguous(), cache, k_d[:, p].contiguous(),
                                       v_d[:, p].contiguous(), W, theta, out=out, lse=lse, workspace=ws,
                                       cache_struct=st)
        if p in check_at:
            outs[p] = (out, lse)
    torch.cuda.synchronize()
    return cache, {p: (host(o), host(l)) for p, (o, l) in outs.items()}


@pytest.mark.parametrize("Hq,Hkv,d,n_pinned,ring_extra,theta", [
    (4, 2, 64, 0, 0, 10000.0),
    (8, 2, 128, 0, 8, 10000.0),     # ring larger than the window
    (4, 4, 64, 5, 0, 10000.0),      # pinned prefix + compressed
    (16, 2, 128, 3, 0, 0.0),        # no rotation
])
def test_compressed_decode_steps_match_oracle(Hq, Hkv, d, n_pinned, ring_extra, theta):
    rng = philox(4000 + Hq + d + n_pinned)
    B, T, W, block = 3, 150, 16, 4
    qb, q = normal_bf16(rng, (B, T, Hq, d))
    kb, k = normal_bf16(rng, (B, T, Hkv, d))
    vb, v = normal_bf16(rng, (B, T, Hkv, d))
    check = sorted(set(list(range(0, T, 7)) + [W - 1, W, W + block - 1, W + block, n_pinned + W + block, T - 1]))
    cache, outs = run_steps(qb, kb, vb, W, block, theta, n_pinned, W + ring_extra, set(check), Hq)
    for p in check:
        want, wlse, ref = oracle.compressed_decode(q[:, p], k, v, p, W, block, theta, n_pinned=n_pinned,
                                                   ring_cap=W + ring_extra)
        got, glse = outs[p]
        assert_close_bf16(got, want, f"position {p}")
        np.testing.assert_allclose(glse, wlse, atol=2e-3, rtol=0)
    # metadata after the last step equals the oracle's cache at T-1
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        np.testing.assert_array_equal(host(getattr(cache.kv, f)), getattr(ref, f), err_msg=f)


def gpu_reference_codes(kb, vb, block, theta, W, ring_cap):
    """The library's bulk entry points on the same tokens: pooled blocks
    (nd_kv_compress_pool) and rotated keys (nd_rope_apply), quantised with
    nd_kv_quant_rows."""
    lib = nd()
    B, T, Hkv, d = kb.shape
    k_d, v_d = dev_bf16(kb), dev_bf16(vb)
    pk, pv = lib.nd_kv_compress_pool(k_d, v_d, block, theta)
    kr = lib.nd_rope_apply(k_d, rope_theta=theta) if theta else k_d

    def q8(x):
        codes = torch.empty(x.shape, dtype=torch.int8, device="cuda")
        scales = torch.empty(x.shape[:-1] + (d // 32,), dtype=torch.float32, device="cuda")
        lib.nd_kv_quant_rows(x.contiguous(), codes, scales)
        return host(codes), host(scales)

    return q8(pk), q8(pv), q8(kr), q8(v_d)


@pytest.mark.parametrize("d", [64, 128])
def test_incremental_pooler_writes_the_bulk_pooler_blocks(d):
    """After T steps from an empty cache (no pinned prefix) every pooled slot
    holds exactly nd_kv_compress_pool's block, quantised, and every ring slot
    exactly the rotated (nd_rope_apply) key of its position, quantised."""
    rng = philox(4100 + d)
    B, T, Hq, Hkv, W, block, theta = 2, 203, 4, 2, 24, 4, 10000.0
    qb, _ = normal_bf16(rng, (B, T, Hq, d))
    kb, _ = normal_bf16(rng, (B, T, Hkv, d))
    vb, _ = normal_bf16(rng, (B, T, Hkv, d))
    cache, _ = run_steps(qb, kb, vb, W, block, theta, 0, W, set(), Hq)
    (pkc, pks), (pvc, pvs), (krc, krs), (vc, vs) = gpu_reference_codes(kb, vb, block, theta, W, W)
    nb = T // block
    kv = cache.kv
    got = {f: host(getattr(kv, f)) for f in ("k_codes", "k_scale", "v_codes", "v_scale")}
    # pooled: slot j of [B][Hkv][slot] vs block j of [B][nb][Hkv]
    np.testing.assert_array_equal(got["k_codes"][:, :, :nb], pkc.transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(got["k_scale"][:, :, :nb], pks.transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(got["v_codes"][:, :, :nb], pvc.transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(got["v_scale"][:, :, :nb], pvs.transpose(0, 2, 1, 3))
    # ring: position t sits in ring slot t % W
    S = kv.sink_cap
    for t in range(T - W, T):
        s = S + t % W
        np.testing.assert_array_equal(got["k_codes"][:, :, s], krc[:, t], err_msg=f"key {t}")
        np.testing.assert_array_equal(got["k_scale"][:, :, s], krs[:, t])
        np.testing.assert_array_equal(got["v_codes"][:, :, s], vc[:, t], err_msg=f"value {t}")


def test_compressed_decode_full_size():
    """The compressed-attention workload (B4 H16 d64, W256, b4, RoPE) decoded
    token by token through all 4096 positions (960 pooled blocks + 256 exact
    keys at the end): outputs at the window edge, the first block arrivals, a
    middle position and the last, against the oracle; pooled codes against
    the bulk pooler."""
    w = compressed()
    B, T, H, d = w["q"].shape
    W, block, theta = w["window"], w["block"], w["rope_theta"]
    check = {W - 1, W + block - 1, W + block, 2000, T - 1}
    cache, outs = run_steps(w["q_bits"], w["k_bits"], w["v_bits"], W, block, theta, 0, W, check, H)
    for p in sorted(check):
        want, wlse, _ = oracle.compressed_decode(w["q"][:, p], w["k"], w["v"], p, W, block, theta)
        got, glse = outs[p]
        assert_close_bf16(got, want, f"position {p}")
        np.testing.assert_allclose(glse, wlse, atol=2e-3, rtol=0)
    (pkc, _), (pvc, _), _, _ = gpu_reference_codes(w["k_bits"], w["v_bits"], block, theta, W, W)
    nb = T // block
    np.testing.assert_array_equal(host(cache.kv.k_codes)[:, :, :nb], pkc.transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(host(cache.kv.v_codes)[:, :, :nb], pvc.transpose(0, 2, 1, 3))
    assert np.all(host(cache.kv.sink_len) == (T - W) // block)


def test_compressed_decode_refuses_bad_shapes():
    lib = nd()
    cache = lib.CompressedCache.empty(2, 2, 64, 8, 16, 4)
    q = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    for W, want in ((17, lib.nd.ND_ERR_INVALID_ARG),   # the window does not fit the ring
                    (0, lib.nd.ND_ERR_INVALID_ARG)):
        with pytest.raises(lib.NDError) as ei:
            lib.nd_compressed_decode_step(q, cache, kn, kn, W, 10000.0)
        assert ei.value.status == want
    bad = lib.CompressedCache.empty(2, 2, 64, 8, 16, 0)   # block 0
    with pytest.raises(lib.NDError):
        lib.nd_compressed_decode_step(q, bad, kn, kn, 16, 10000.0)
