"""Host checks of the fp32 facts the CUDA quantisers rely on.

The cache codec is scale = amax / 127 and code = clamp(rint(x / scale), +-127)
with IEEE fp32 divides ("How the 256-Token Sliding Window Works with Tools as
KV Sinks in Needle", section "Effective KV Window": int8 codes with one fp32
scale per 32 channels).  The kernels avoid the divide on almost every element:
p = x * fl(1 / scale) is rounded instead of the quotient unless p lies within
1e-4 of a half-integer (or the scale is below 1e-30), and the handoff's
quantiser rounds p by adding and subtracting 1.5 * 2^23 and takes the code's
byte from the sum, with no clamp outside that band.  numpy's float32 multiply,
divide and add are correctly rounded (round to nearest even), as the GPU's
__fmul_rn / __fdiv_rn / __frcp_rn / __fadd_rn are, so these checks hold for
the device arithmetic too.
"""
import numpy as np

MAGIC = np.float32(12582912.0)  # 1.5 * 2^23


def _magic_round(p):
    t = (p + MAGIC).astype(np.float32)
    return t, (t - MAGIC).astype(np.float32)


def test_magic_number_rounding_is_rint_near_every_half_integer():
    """Every float32 within 2^-6 of k + 1/2 or of k, |k| <= 128: the sum's
    value and low byte are rint(p) (ties to even) and its two's-complement
    byte."""
    pts = []
    for k in range(-129, 129):
        for c in (k, k + 0.5):
            lo = np.float32(c - 2.0 ** -6)
            hi = np.float32(c + 2.0 ** -6)
            # every float32 in [lo, hi]: walk the ordered bit patterns
            a, b = np.array([lo, hi], np.float32).view(np.int32)
            if lo < 0 <= hi or lo <= 0 < hi:
                continue  # the band around 0 is covered by the random sample
            if lo < 0:
                a, b = b, a
            bits = np.arange(a, b + 1, dtype=np.int64).astype(np.int32)
            pts.append(bits.view(np.float32))
    p = np.concatenate(pts)
    t, r = _magic_round(p)
    np.testing.assert_array_equal(r, np.rint(p))
    byte = (t.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8)
    np.testing.assert_array_equal(byte.astype(np.int32), np.rint(p).astype(np.int32).astype(np.int8))


def test_magic_number_rounding_on_a_random_sample():
    rng = np.random.default_rng(7)
    p = rng.uniform(-128.0, 128.0, 2_000_000).astype(np.float32)
    p = np.concatenate([p, np.float32([0.0, -0.0, 0.5, -0.5, 1.5, -1.5, 127.5, -127.5, 2.0 ** -149])])
    t, r = _magic_round(p)
    np.testing.assert_array_equal(r, np.rint(p))
    byte = (t.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8)
    np.testing.assert_array_equal(byte.astype(np.int32), np.rint(p).astype(np.int32).astype(np.int8))


def test_fast_path_code_equals_the_quotient_code_and_needs_no_clamp():
    """Outside the 1e-4 band around half-integers, with a normal scale,
    rint(x * fl(1/scale)) = rint(fl(x / scale)) and |x * fl(1/scale)| < 127.5,
    for groups of every magnitude (amax from 2^-100 to 2^100)."""
    rng = np.random.default_rng(11)
    n = 400_000
    amax = (2.0 ** rng.uniform(-100, 100, n)).astype(np.float32)
    frac = rng.uniform(-1.0, 1.0, n).astype(np.float32)
    x = (frac * amax).astype(np.float32)
    x[::7] = amax[::7]                          # the group maximum itself
    x[1::7] = -amax[1::7]
    scale = (amax / np.float32(127.0)).astype(np.float32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    p = (x * inv).astype(np.float32)
    r = np.rint(p)
    fast = (np.abs(np.abs(p - r) - np.float32(0.5)) > np.float32(1e-4)) & (scale >= np.float32(1e-30))
    normal = scale >= np.float32(1e-30)
    assert fast[normal].mean() > 0.99           # the band itself is rare
    q = np.rint((x / scale).astype(np.float32))
    np.testing.assert_array_equal(r[fast], q[fast])
    assert np.all(np.abs(p[fast]) < 127.5)
    assert np.all(np.abs(r[fast]) <= 127)
