"""GPU parity: int8 group-32 codec, fused quantise-and-append, and decode,
against the fp64 oracle (codes and cache metadata bit-exact; decode outputs
within max-abs 2e-2 / mean-abs 2e-3, the bf16 tolerance)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close_bf16, dev, dev_bf16, host, need_gpu, no_device_errors
from workloads import (bf16_bits_to_f32, decode_b64, decode_cache, decode_sweep, normal_bf16, philox,
                       random_codes, to_bf16_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    no_device_errors()


def nd():
    import sliding_window_kv_swa_gb300 as m
    return m


# ---------------------------------------------------------------- codec

@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_quant_rows_bit_exact(d):
    rng = philox(200 + d)
    n = 3001
    x = rng.standard_normal((n, d), dtype=np.float32) * rng.uniform(1e-3, 1e3, (n, 1)).astype(np.float32)
    x[5] = 0.0                                    # zero group -> scale 0
    x[6, :32] = 1e-30                             # tiny values (bf16 subnormal range)
    bits = to_bf16_bits(x)
    codes = torch.empty((n, d), dtype=torch.int8, device="cuda")
    scales = torch.empty((n, d // 32), dtype=torch.float32, device="cuda")
    nd().nd_kv_quant_rows(dev_bf16(bits), codes, scales)
    wc, ws = oracle.quant_g32(bf16_bits_to_f32(bits))
    np.testing.assert_array_equal(host(codes), wc)
    np.testing.assert_array_equal(host(scales).view(np.uint32), ws.view(np.uint32))


def test_quant_rows_quotients_at_and_beside_half_integers():
    """Groups whose quotients x / scale sit exactly on half-integers (ties to
    even) and one or two bf16 steps either side of them, at several scales:
    the kernels' rounding near these boundaries must give the oracle's codes
    (fp32 IEEE divide, rint) bit for bit."""
    rows = []
    for k in (-20, -3, 0, 5, 17):
        sc = 2.0 ** k
        for n in range(-127, 127, 3):
            base = (n + 0.5) * sc
            vals = [base]
            b = to_bf16_bits(np.array([base], np.float32)).astype(np.int32)[0]
            for dlt in (-2, -1, 1, 2):
                vals.append(float(bf16_bits_to_f32(np.array([b + dlt], np.uint16))[0]))
            row = np.zeros(32, np.float32)
            row[0] = 127.0 * sc              # amax: scale = 2^k exactly
            row[1:1 + len(vals)] = vals
            row[6:] = np.linspace(-126.0, 126.0, 26, dtype=np.float32) * sc
            rows.append(row)
    while len(rows) % 4:
        rows.append(rows[0])
    x = np.stack(rows).reshape(-1, 128)
    bits = to_bf16_bits(x)
    n = x.shape[0]
    codes = torch.empty((n, 128), dtype=torch.int8, device="cuda")
    scales = torch.empty((n, 4), dtype=torch.float32, device="cuda")
    nd().nd_kv_quant_rows(dev_bf16(bits), codes, scales)
    wc, ws = oracle.quant_g32(bf16_bits_to_f32(bits))
    np.testing.assert_array_equal(host(codes), wc)
    np.testing.assert_array_equal(host(scales).view(np.uint32), ws.view(np.uint32))


def test_quant_rows_golden_ties():
    from test_oracle_attention import read_codec_fixture
    groups = read_codec_fixture()
    x = np.array([g["x"] for g in groups], np.float32).reshape(1, -1)
    codes = torch.empty((1, 128), dtype=torch.int8, device="cuda")
    scales = torch.empty((1, 4), dtype=torch.float32, device="cuda")
    nd().nd_kv_quant_rows(dev_bf16(to_bf16_bits(x)), codes, scales)
    np.testing.assert_array_equal(host(codes).reshape(-1), np.array([g["code"] for g in groups]).reshape(-1))


@pytest.mark.parametrize("d", [64, 128])
def test_append_sequence_matches_oracle(d):
    """Sinks first, then the ring fills, wraps twice; every step bit-exact."""
    B, Hkv, S, W = 5, 3, 4, 8
    rng = philox(300 + d)
    ref = oracle.Cache(B, Hkv, d, S, W)
    cache = nd().KVCache.empty(B, Hkv, d, S, W)
    for step in range(S + 2 * W + 3):
        to_sink = step < S
        kb, kf = normal_bf16(rng, (B, Hkv, d))
        vb, vf = normal_bf16(rng, (B, Hkv, d))
        nd().nd_kv_append_quant(cache, dev_bf16(kb), dev_bf16(vb), to_sink)
        assert oracle.kv_append(ref, kf, vf, to_sink) == 0
        for name in ("k_codes", "v_codes", "k_scale", "v_scale", "sink_len", "ring_start", "ring_len", "seq_len"):
            np.testing.assert_array_equal(host(getattr(cache, name)), getattr(ref, name), err_msg=f"{name} step {step}")


def test_rejected_sink_append_sets_flag_and_writes_nothing():
    B, Hkv, d, S, W = 2, 1, 64, 2, 4
    cache = nd().KVCache.empty(B, Hkv, d, S, W)
    rng = philox(310)
    kb, _ = normal_bf16(rng, (B, Hkv, d))
    nd().nd_kv_append_quant(cache, dev_bf16(kb), dev_bf16(kb), False)   # ring token first
    before = host(cache.k_codes).copy()
    nd().nd_kv_append_quant(cache, dev_bf16(kb), dev_bf16(kb), True)    # then a sink: rejected
    assert nd().nd_device_errors(clear=True) == 2
    np.testing.assert_array_equal(host(cache.k_codes), before)
    np.testing.assert_array_equal(host(cache.sink_len), [0, 0])
    np.testing.assert_array_equal(host(cache.seq_len), [1, 1])


# ---------------------------------------------------------------- decode

def device_cache(ref: "oracle.Cache"):
    c = nd().KVCache(dev(ref.k_codes), dev(ref.v_codes), dev(ref.k_scale), dev(ref.v_scale),
                     dev(ref.sink_len), dev(ref.ring_start), dev(ref.ring_len), dev(ref.seq_len),
                     ref.sink_cap, ref.ring_cap)
    return c


def oracle_cache(w, S, W):
    B, Hkv, ns, d = w["k"].shape
    ref = oracle.Cache(B, Hkv, d, S, W)
    ref.k_codes[...], ref.k_scale[...] = oracle.quant_g32(w["k"])
    ref.v_codes[...], ref.v_scale[...] = oracle.quant_g32(w["v"])
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        getattr(ref, f)[...] = w[f]
    return ref


def run_decode(ref, q_bits, window, lse=True):
    B, Hq, d = q_bits.shape
    cache = device_cache(ref)
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((B, Hq), dtype=torch.float32, device="cuda") if lse else None
    nd().nd_swa_sink_decode(dev_bf16(q_bits), cache, window, out=out, lse=l)
    return host(out), (host(l) if lse else None)


def test_decode_b64_matches_oracle():
    w = decode_b64()
    ref = oracle_cache(w, 64, 256)
    got, lse = run_decode(ref, w["q_bits"], 256)
    want, wlse = oracle.decode(w["q"], ref, 256)
    assert_close_bf16(got, want, "decode B64")
    np.testing.assert_allclose(lse, wlse, atol=2e-3, rtol=0)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 1, 64), (8, 8, 128), (16, 2, 128), (6, 2, 64), (32, 8, 128)])
def test_decode_partial_rings_and_windows(Hq, Hkv, d):
    rng = philox(400 + Hq + d)
    S, W, B = 24, 40, 7
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=401 + Hq, full=False)
    ref = oracle_cache(w, S, W)
    # per-sequence variety: fewer sinks, empty ring, wrapped ring
    ref.sink_len[:] = [24, 0, 5, 24, 17, 1, 24]
    ref.ring_len[:] = [40, 13, 0, 40, 1, 40, 27]
    ref.ring_start[:] = [7, 0, 0, 39, 0, 0, 0]
    ref.seq_len[:] = ref.sink_len + ref.ring_len + np.array([7, 0, 0, 39, 0, 0, 0])
    for window in (W, 17, 1, 3 * W):
        got, lse = run_decode(ref, w["q_bits"], window)
        want, wlse = oracle.decode(w["q"], ref, window)
        assert_close_bf16(got, want, f"decode window {window}")
        np.testing.assert_allclose(lse, wlse, atol=2e-3, rtol=0)


def test_decode_empty_cache_gives_zero_and_neg_inf():
    B, Hq, Hkv, d, S, W = 3, 4, 1, 64, 8, 16
    ref = oracle.Cache(B, Hkv, d, S, W)
    q_bits, _ = normal_bf16(philox(410), (B, Hq, d))
    got, lse = run_decode(ref, q_bits, W)
    assert np.all(got == 0) and np.all(np.isneginf(lse))


def test_decode_invariant_to_ring_rotation():
    S, W, Hq, Hkv, d = 16, 64, 8, 2, 128
    w = decode_cache(2, Hq, Hkv, d, S, W, seed=420, full=True)
    ref = oracle_cache(w, S, W)
    base, _ = run_decode(ref, w["q_bits"], W)
    for shift in (1, 17, 63):
        r2 = ref.copy()
        for arr in (r2.k_codes, r2.v_codes, r2.k_scale, r2.v_scale):
            arr[:, :, S:] = np.roll(arr[:, :, S:], shift, axis=2)
        r2.ring_start[:] = (ref.ring_start + shift) % W
        got, _ = run_decode(r2, w["q_bits"], W)
        assert np.abs(got - base).max() <= 4e-3   # summation order only


def test_decode_large_magnitudes_and_tiny_values():
    """Power-of-two pre-scaling keeps fp16 operands exact at any magnitude."""
    S, W, Hq, Hkv, d = 8, 32, 4, 1, 64
    for mag in (1e-6, 1e-2, 1e3):
        w = decode_cache(2, Hq, Hkv, d, S, W, seed=430, full=True)
        w["k"] = bf16_bits_to_f32(to_bf16_bits(w["k"] * mag))
        w["v"] = bf16_bits_to_f32(to_bf16_bits(w["v"] * mag))
        q_bits = to_bf16_bits(w["q"] * (1.0 / max(mag, 1e-3)))
        ref = oracle_cache(w, S, W)
        got, _ = run_decode(ref, q_bits, W, lse=False)
        want, _ = oracle.decode(bf16_bits_to_f32(q_bits), ref, W)
        err = np.abs(got - want).max() / max(np.abs(want).max(), 1e-30)
        assert err < 1e-2, (mag, err)


@pytest.mark.parametrize("B", [32, 64, 128, 512])
def test_decode_sweep_full_size_all_sequences(B):
    """Configuration of the large-batch sweep (Hq32 Hkv8 d128, 1024 sinks + 256
    ring) at full size, in the bench's launch configuration: every sequence
    (out and lse) against the oracle.  B64 and B128 leave a partial last wave
    of (sequence, KV head) pairs, B32 less than one wave."""
    rng = philox(500 + B)
    Hq, Hkv, d, S, W = 32, 8, 128, 1024, 256
    kc, ks, vc, vs = random_codes(rng, B, Hkv, S + W, d)
    ring_start = rng.integers(0, W, size=B).astype(np.int32)
    meta = dict(sink_len=np.full(B, S, np.int32), ring_start=ring_start,
                ring_len=np.full(B, W, np.int32), seq_len=(S + W + ring_start).astype(np.int32))
    q_bits, q = normal_bf16(rng, (B, Hq, d))
    cache = nd().KVCache(dev(kc), dev(vc), dev(ks), dev(vs), dev(meta["sink_len"]), dev(meta["ring_start"]),
                         dev(meta["ring_len"]), dev(meta["seq_len"]), S, W)
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    nd().nd_swa_sink_decode(dev_bf16(q_bits), cache, W, out=out, lse=lse)
    got, got_lse = host(out), host(lse)
    del cache, out
    ref = oracle.Cache.__new__(oracle.Cache)
    ref.B, ref.Hkv, ref.d, ref.sink_cap, ref.ring_cap = B, Hkv, d, S, W
    ref.k_codes, ref.k_scale, ref.v_codes, ref.v_scale = kc, ks, vc, vs
    for f in meta:
        setattr(ref, f, meta[f])
    want, wlse = oracle.decode(q, ref, W)
    assert_close_bf16(got, want, f"decode sweep B{B}")
    for b in range(0, B, 64):   # and per block of sequences
        assert_close_bf16(got[b:b + 64], want[b:b + 64], f"sequences {b}..{b + 63}")
    np.testing.assert_allclose(got_lse, wlse, atol=2e-3, rtol=0)


def test_append_then_decode_step():
    """The decode-sweep step: quantise-and-append one token, then attend."""
    B, Hq, Hkv, d, S, W = 6, 32, 8, 128, 64, 32
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=600, full=True)
    ref = oracle_cache(w, S, W)
    cache = device_cache(ref)
    rng = philox(601)
    for step in range(3):
        kb, kf = normal_bf16(rng, (B, Hkv, d))
        vb, vf = normal_bf16(rng, (B, Hkv, d))
        qb, qf = normal_bf16(rng, (B, Hq, d))
        nd().nd_kv_append_quant(cache, dev_bf16(kb), dev_bf16(vb), False)
        oracle.kv_append(ref, kf, vf, False)
        out = nd().nd_swa_sink_decode(dev_bf16(qb), cache, W)
        want, _ = oracle.decode(qf, ref, W)
        assert_close_bf16(host(out), want, f"step {step}")
    np.testing.assert_array_equal(host(cache.k_codes), ref.k_codes)


@pytest.mark.parametrize("B,Hq,Hkv,d,S,W,fill", [
    (10, 32, 8, 128, 64, 32, "full"),    # 8 KV heads: append and decode as two launches
    (20, 16, 4, 128, 64, 32, "full"),    # one cluster of 4 KV heads per sequence: fused
    (64, 8, 2, 64, 64, 256, "full"),     # the decode-step configuration: fused
    (5, 4, 1, 64, 24, 40, "partial"),    # rings still filling, then wrapping
    (1, 16, 8, 128, 64, 192, "partial"),  # one sequence: 4-way split x 8 KV heads, two launches
])
def test_decode_step_matches_append_then_decode(B, Hq, Hkv, d, S, W, fill):
    """nd_swa_sink_decode_step (append the token, then attend with it) against
    the oracle's append followed by its decode: output within the bf16
    tolerance; codes, scales and metadata bit-exact after every step."""
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=700 + B + d, full=(fill == "full"))
    ref = oracle_cache(w, S, W)
    if fill == "partial":
        ref.ring_len[:] = np.arange(B) % 3
        ref.ring_start[:] = 0
        ref.seq_len[:] = ref.sink_len + ref.ring_len
    cache = device_cache(ref)
    rng = philox(701 + B)
    steps = W + 3 if fill == "partial" else 3
    for step in range(steps):
        kb, kf = normal_bf16(rng, (B, Hkv, d))
        vb, vf = normal_bf16(rng, (B, Hkv, d))
        qb, qf = normal_bf16(rng, (B, Hq, d))
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        out = nd().nd_swa_sink_decode_step(dev_bf16(qb), cache, dev_bf16(kb), dev_bf16(vb), W, lse=lse)
        oracle.kv_append(ref, kf, vf, False)
        if step % 7 == 0 or step == steps - 1:
            want, wlse = oracle.decode(qf, ref, W)
            assert_close_bf16(host(out), want, f"step {step}")
            np.testing.assert_allclose(host(lse), wlse, atol=2e-3, rtol=0)
            for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
                np.testing.assert_array_equal(host(getattr(cache, f)), getattr(ref, f), err_msg=f)
    np.testing.assert_array_equal(host(cache.k_codes), ref.k_codes)
    np.testing.assert_array_equal(host(cache.v_codes), ref.v_codes)
    np.testing.assert_array_equal(host(cache.k_scale), ref.k_scale)
    np.testing.assert_array_equal(host(cache.v_scale), ref.v_scale)


@pytest.mark.parametrize("B,Hq,Hkv,d,S,W,packed", [
    (64, 8, 2, 64, 64, 256, False),   # fused step
    (64, 8, 2, 64, 64, 256, True),    # packed host buffers: one copy each way
    (10, 32, 8, 128, 64, 32, False),  # append and decode as two launches
    (10, 32, 8, 128, 64, 32, True),
    (3, 3, 1, 64, 8, 16, False),      # lse of 36 bytes, written in place
    (3, 3, 1, 64, 8, 16, True),
])
def test_decode_step_host_buffers(B, Hq, Hkv, d, S, W, packed):
    """nd_swa_sink_decode_step_host (separate host buffers) and
    nd_swa_sink_decode_step_host_packed (q | k_new | v_new in one host
    allocation, out | lse in another): the copies are enqueued by the call;
    same results as the oracle's append + decode, cache bit-exact."""
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=760 + B + d, full=True)
    ref = oracle_cache(w, S, W)
    cache = device_cache(ref)
    st = cache.struct()
    ws = torch.empty(nd().nd_swa_sink_decode_step_host_workspace_size(B, Hq, Hkv, d, S + W),
                     dtype=torch.uint8, device="cuda")
    rng = philox(761 + B)
    nq, nk = B * Hq * d, B * Hkv * d
    if packed:
        obuf = torch.empty(nq * 2 + B * Hq * 4, dtype=torch.uint8).pin_memory()
        out_h = obuf[:nq * 2].view(torch.bfloat16).view(B, Hq, d)
        lse_h = obuf[nq * 2:].view(torch.float32).view(B, Hq)
    else:
        out_h = torch.empty((B, Hq, d), dtype=torch.bfloat16).pin_memory()
        lse_h = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
    pin = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()
    for step in range(3):
        kb, kf = normal_bf16(rng, (B, Hkv, d))
        vb, vf = normal_bf16(rng, (B, Hkv, d))
        qb, qf = normal_bf16(rng, (B, Hq, d))
        if packed:
            inp = pin(np.concatenate([np.ascontiguousarray(x).view(np.int16).reshape(-1) for x in (qb, kb, vb)]))
            nd().nd_swa_sink_decode_step_host_packed(inp, cache, Hq, W, obuf, with_lse=True, workspace=ws,
                                                     cache_struct=st)
        else:
            nd().nd_swa_sink_decode_step_host(pin(qb), cache, pin(kb), pin(vb), W, out_h, lse_host=lse_h,
                                              workspace=ws, cache_struct=st)
        torch.cuda.current_stream().synchronize()
        oracle.kv_append(ref, kf, vf, False)
        want, wlse = oracle.decode(qf, ref, W)
        assert_close_bf16(out_h.float().numpy(), want, f"host step {step}")
        np.testing.assert_allclose(lse_h.numpy(), wlse, atol=2e-3, rtol=0)
    np.testing.assert_array_equal(host(cache.k_codes), ref.k_codes)
    np.testing.assert_array_equal(host(cache.v_scale), ref.v_scale)
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        np.testing.assert_array_equal(host(getattr(cache, f)), getattr(ref, f), err_msg=f)


@pytest.mark.parametrize("B,Hq,Hkv,d,S,W", [
    (64, 8, 2, 64, 64, 256),    # fused step, one CTA per SM (early trigger of the next step)
    (10, 32, 8, 128, 64, 32),   # append, then the decode as a dependent launch
    (1, 16, 8, 128, 64, 192),   # split decode + combine after the append
])
def test_decode_steps_back_to_back(B, Hq, Hkv, d, S, W):
    """Steps enqueued back to back with every input already on the device and
    no synchronisation in between, so each step's kernels are scheduled while
    the previous step's run (dependent launches): every step must still see
    the token the step before appended.  Outputs are kept per step and
    checked against the oracle's sequence afterwards."""
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=790 + B + d, full=True)
    ref = oracle_cache(w, S, W)
    cache = device_cache(ref)
    rng = philox(791 + B)
    n = 6
    toks = [(normal_bf16(rng, (B, Hkv, d)), normal_bf16(rng, (B, Hkv, d)), normal_bf16(rng, (B, Hq, d)))
            for _ in range(n)]
    dev_in = [(dev_bf16(kb), dev_bf16(vb), dev_bf16(qb)) for (kb, _), (vb, _), (qb, _) in toks]
    outs = [torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    ws = torch.empty(max(nd().nd_swa_sink_decode_workspace_size(B, Hq, Hkv, d, S + W), 16), dtype=torch.uint8,
                     device="cuda")
    torch.cuda.synchronize()
    for i in range(n):
        k_d, v_d, q_d = dev_in[i]
        nd().nd_swa_sink_decode_step(q_d, cache, k_d, v_d, W, out=outs[i], workspace=ws)
    torch.cuda.synchronize()
    for i, ((_, kf), (_, vf), (_, qf)) in enumerate(toks):
        oracle.kv_append(ref, kf, vf, False)
        want, _ = oracle.decode(qf, ref, W)
        assert_close_bf16(host(outs[i]), want, f"step {i}")
    np.testing.assert_array_equal(host(cache.k_codes), ref.k_codes)
    for f in ("sink_len", "ring_start", "ring_len", "seq_len"):
        np.testing.assert_array_equal(host(getattr(cache, f)), getattr(ref, f), err_msg=f)


def test_decode_steps_host_packed_back_to_back():
    """The packed host-buffer step (the step's kernels read and write the
    page-locked buffers in place) for several steps without synchronisation
    in between, each step on its own buffers."""
    B, Hq, Hkv, d, S, W = 64, 8, 2, 64, 64, 256
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=795, full=True)
    ref = oracle_cache(w, S, W)
    cache = device_cache(ref)
    st = cache.struct()
    ws = torch.empty(nd().nd_swa_sink_decode_step_host_workspace_size(B, Hq, Hkv, d, S + W),
                     dtype=torch.uint8, device="cuda")
    rng = philox(796)
    n = 5
    toks = [(normal_bf16(rng, (B, Hkv, d)), normal_bf16(rng, (B, Hkv, d)), normal_bf16(rng, (B, Hq, d)))
            for _ in range(n)]
    ins = [torch.from_numpy(np.concatenate([np.ascontiguousarray(x).view(np.int16).reshape(-1)
                                            for x in (qb, kb, vb)])).view(torch.bfloat16).pin_memory()
           for (kb, _), (vb, _), (qb, _) in toks]
    outs = [torch.empty((B, Hq, d), dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        nd().nd_swa_sink_decode_step_host_packed(ins[i], cache, Hq, W, outs[i], workspace=ws, cache_struct=st)
    torch.cuda.synchronize()
    for i, ((_, kf), (_, vf), (_, qf)) in enumerate(toks):
        oracle.kv_append(ref, kf, vf, False)
        want, _ = oracle.decode(qf, ref, W)
        assert_close_bf16(outs[i].float().numpy(), want, f"step {i}")


@pytest.mark.parametrize("packed", [False, True])
def test_decode_step_host_pageable_and_no_lse(packed):
    """Host buffers that are not page-locked take the copy-engine path
    (cudaMemcpyAsync) instead of being accessed in place; the packed form without
    lse copies the output alone.  Same results as the oracle either way."""
    B, Hq, Hkv, d, S, W = 8, 8, 2, 64, 16, 48
    w = decode_cache(B, Hq, Hkv, d, S, W, seed=798 + packed, full=True)
    ref = oracle_cache(w, S, W)
    cache = device_cache(ref)
    ws = torch.empty(nd().nd_swa_sink_decode_step_host_workspace_size(B, Hq, Hkv, d, S + W),
                     dtype=torch.uint8, device="cuda")
    rng = philox(799 + packed)
    for step in range(2):
        kb, kf = normal_bf16(rng, (B, Hkv, d))
        vb, vf = normal_bf16(rng, (B, Hkv, d))
        qb, qf = normal_bf16(rng, (B, Hq, d))
        as_t = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        if packed:
            inp = as_t(np.concatenate([np.ascontiguousarray(x).view(np.int16).reshape(-1) for x in (qb, kb, vb)]))
            out_h = torch.empty((B, Hq, d), dtype=torch.bfloat16)
            nd().nd_swa_sink_decode_step_host_packed(inp, cache, Hq, W, out_h, with_lse=False, workspace=ws)
        else:
            out_h = torch.empty((B, Hq, d), dtype=torch.bfloat16)
            lse_h = torch.empty((B, Hq), dtype=torch.float32)
            nd().nd_swa_sink_decode_step_host(as_t(qb), cache, as_t(kb), as_t(vb), W, out_h, lse_host=lse_h,
                                              workspace=ws)
        torch.cuda.current_stream().synchronize()
        oracle.kv_append(ref, kf, vf, False)
        want, wlse = oracle.decode(qf, ref, W)
        assert_close_bf16(out_h.float().numpy(), want, f"step {step}")
        if not packed:
            np.testing.assert_allclose(lse_h.numpy(), wlse, atol=2e-3, rtol=0)
    np.testing.assert_array_equal(host(cache.k_codes), ref.k_codes)
