"""fp64 CPU oracle for sliding-window + KV-sink attention (test infrastructure).

This package is TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import it.  The product library never
does, and it shares no code with the CUDA path.  The arithmetic lives in
``nd_oracle.c`` (plain C, fp64, explicit dense masks); this module compiles it
with gcc and marshals numpy arrays in and out.  Each wrapper names the page
section its C function follows.

Sources: "How the 256-Token Sliding Window Works with Tools as KV Sinks in
Needle" (mask, budget), "256-token滑动窗口+KV sink：Needle 2工具钉住机制源码分析"
(decode mask, budget constants), "Compressed attention and the copy probe"
(compressed mask, pooling, midpoint rotation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnd_oracle.so")

# The codec must be compiled without FMA contraction or fast-math so that the
# fp32 divide and rint decide every int8 code exactly as written.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wno-unknown-pragmas"]

_lib = None


def build(force: bool = False) -> str:
    """Compile nd_oracle.c into a shared library next to it; returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if force or not fresh:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        D = ctypes.c_double
        sig = {
            "ndo_num_threads": (I, []),
            "ndo_causal_packing_mask": (None, [I, I, P, P, I, P]),
            "ndo_decode_keep": (None, [I, L, P, P, I, P]),
            "ndo_window_mask": (None, [I, I, P]),
            "ndo_compressed_mask": (None, [I, I, I, P]),
            "ndo_attention": (None, [I, I, I, I, I, I, P, P, P, P, L, I, P, P, P]),
            "ndo_quant_g32": (None, [I, I, P, P, P]),
            "ndo_kv_append": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I]),
            "ndo_slot_positions": (None, [I, I, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, P, P]),
            "ndo_decode": (None, [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I, P, P]),
            "ndo_pool_blocks": (None, [I, I, I, I, I, P, P]),
            "ndo_rope": (None, [I, I, I, I, P, P, D, P]),
            "ndo_compress": (None, [I, I, I, I, I, D, I, P, P, P, P, P, P]),
            "ndo_kv_budget_window": (L, [L, L, L, L, L, L, L]),
            "ndo_effective_kv_window": (L, [L, L]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().ndo_num_threads())


# --------------------------------------------------------------------------
# Masks
# --------------------------------------------------------------------------

def causal_packing_mask(seg_ids, prefix=None, window: int = 0) -> np.ndarray:
    """make_causal_packing_mask ("KV Sinks for Tools"): bool [B, T, T]."""
    seg = _c(seg_ids, np.int32)
    B, T = seg.shape
    pre = None if prefix is None else _c(np.asarray(prefix) > 0, np.uint8)
    out = np.empty((B, T, T), np.uint8)
    _load().ndo_causal_packing_mask(B, T, _ptr(seg), _ptr(pre), int(window), _ptr(out))
    return out.astype(bool)


def decode_keep(qpos: int, kpos, sink=None, kv_window: int = 0) -> np.ndarray:
    """Decode mask ("256-token 滑动窗口：源码走读"): bool [n_keys]."""
    kp = _c(kpos, np.int64)
    sk = None if sink is None else _c(np.asarray(sink) != 0, np.uint8)
    out = np.empty(kp.shape[0], np.uint8)
    _load().ndo_decode_keep(kp.shape[0], int(qpos), _ptr(kp), _ptr(sk), int(kv_window), _ptr(out))
    return out.astype(bool)


def window_mask(length: int, window: int) -> np.ndarray:
    """attention_mask(length, window, 0) as read here: causal sliding window."""
    out = np.empty((length, length), np.uint8)
    _load().ndo_window_mask(int(length), int(window), _ptr(out))
    return out.astype(bool)


def compressed_mask(length: int, window: int, block: int) -> np.ndarray:
    """compressed_mask ("Two kinds of columns"): bool [T, T//block + T]."""
    out = np.empty((length, length // block + length), np.uint8)
    _load().ndo_compressed_mask(int(length), int(window), int(block), _ptr(out))
    return out.astype(bool)


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def attention(q, k, v, mask, rows=None):
    """Dense masked softmax attention in fp64 with contiguous GQA groups.

    q [B,Tq,Hq,d], k/v [B,Tk,Hkv,d], mask [B,Tq,Tk] or [Tq,Tk] (shared by the
    batch).  rows: None, or an int array [n,2] of (b, t) rows to compute.
    Returns (out, lse): out [B,Tq,Hq,d] (or [n,Hq,d]), lse [B,Tq,Hq] (or [n,Hq]).
    """
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    B, Tq, Hq, d = q.shape
    _, Tk, Hkv, _ = k.shape
    assert Hq % Hkv == 0
    m = _c(np.asarray(mask, dtype=bool), np.uint8)
    bstride = 0 if m.ndim == 2 else Tq * Tk
    if rows is None:
        out = np.empty((B, Tq, Hq, d), np.float64)
        lse = np.empty((B, Tq, Hq), np.float64)
        n, rp = 0, None
    else:
        rp = _c(rows, np.int32).reshape(-1, 2)
        n = rp.shape[0]
        out = np.empty((n, Hq, d), np.float64)
        lse = np.empty((n, Hq), np.float64)
    _load().ndo_attention(B, Tq, Tk, Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v), _ptr(m),
                          bstride, n, _ptr(rp), _ptr(out), _ptr(lse))
    return out, lse


def swa_sink_prefill(q, k, v, seg_ids, sink=None, window: int = 0,
                     rope_theta: float = 0.0, rows=None):
    """Prefill: rotate q and k at their packed positions (when rope_theta is
    non-zero), build make_causal_packing_mask, and attend.  GQA by contiguous
    groups.  Returns (out, lse) as :func:`attention`."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    B, T = q.shape[:2]
    if rope_theta:
        pos = np.arange(T, dtype=np.int64)
        q = rope(q, pos, rope_theta)
        k = rope(k, pos, rope_theta)
    mask = causal_packing_mask(seg_ids, sink, window)
    return attention(q, k, v, mask, rows)


def compressed_prefill(q, k, v, window: int, block: int, rope_theta: float = 0.0,
                       rows=None):
    """Compressed attention ("Two kinds of columns", "Pool before rotating"):
    _compress, then one softmax over [pooled blocks, exact windowed keys]."""
    qr, kk, vv = compress(q, k, v, block, rope_theta)
    T = q.shape[1]
    mask = compressed_mask(T, window, block)
    return attention(qr, kk, vv, mask, rows)


def compressed_prefill_pinned(q, k, v, window: int, block: int, n_pinned: int,
                              rope_theta: float = 0.0, rows=None):
    """Compressed attention with a pinned prefix ("Compressed attention and
    the copy probe" with the sink prefix of "KV Sinks for Tools"; the reading
    used by the compressed decode): keys 0..n_pinned-1 are exact keys visible
    at any distance; pooled block j covers positions n_pinned + j*block ..
    + block-1 (mean before rotation, rotated at n_pinned + j*block +
    block//2) and is visible to query t iff (j+1)*block <= t - window + 1 -
    n_pinned; other keys k are visible iff k <= t and t - k < window.  One
    softmax over [pooled blocks, exact keys].  Returns (out, lse) as
    :func:`attention`."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    B, T, Hq, d = q.shape
    pos = np.arange(T)
    qr = rope(q, pos, rope_theta) if rope_theta else q
    kr = rope(k, pos, rope_theta) if rope_theta else k
    nb = (T - n_pinned) // block
    pk = pool_blocks(k[:, n_pinned:n_pinned + nb * block], block) if nb else np.zeros((B, 0) + k.shape[2:])
    pv = pool_blocks(v[:, n_pinned:n_pinned + nb * block], block) if nb else np.zeros((B, 0) + v.shape[2:])
    if nb and rope_theta:
        pk = rope(pk, n_pinned + np.arange(nb) * block + block // 2, rope_theta)
    t = pos[:, None]
    j = np.arange(nb)[None, :]
    pooled_vis = (j + 1) * block <= t - window + 1 - n_pinned
    kk = pos[None, :]
    exact_vis = (kk <= t) & ((t - kk < window) | (kk < n_pinned))
    mask = np.concatenate([pooled_vis, exact_vis], axis=1)
    return attention(qr, np.concatenate([pk, kr], axis=1), np.concatenate([pv, v], axis=1), mask, rows)


# --------------------------------------------------------------------------
# int8 group-32 codec and the bounded cache
# --------------------------------------------------------------------------

def quant_g32(x):
    """Quantise fp32 [..., d] (d % 32 == 0) -> (int8 codes [..., d], fp32
    scales [..., d//32]): symmetric absmax/127, fp32 divide, rint, clamp."""
    x = _c(x, np.float32)
    d = x.shape[-1]
    assert d % 32 == 0
    n = x.size // d
    codes = np.empty(x.shape, np.int8)
    scales = np.empty(x.shape[:-1] + (d // 32,), np.float32)
    _load().ndo_quant_g32(n, d, _ptr(x), _ptr(codes), _ptr(scales))
    return codes, scales


def dequant_g32(codes, scales) -> np.ndarray:
    """code * scale in fp64 (exact)."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    s = np.repeat(np.asarray(scales, np.float64), 32, axis=-1)
    assert s.shape[-1] == d
    return codes.astype(np.float64) * s


class Cache:
    """The bounded cache in the library's documented layout, as numpy arrays.

    codes int8 [B][Hkv][sink_cap+ring_cap][d], scales fp32 [...][d/32];
    per-sequence int32 sink_len, ring_start, ring_len, seq_len.
    """

    def __init__(self, B, Hkv, d, sink_cap, ring_cap):
        self.B, self.Hkv, self.d = B, Hkv, d
        self.sink_cap, self.ring_cap = sink_cap, ring_cap
        ns = sink_cap + ring_cap
        self.k_codes = np.zeros((B, Hkv, ns, d), np.int8)
        self.v_codes = np.zeros((B, Hkv, ns, d), np.int8)
        self.k_scale = np.zeros((B, Hkv, ns, d // 32), np.float32)
        self.v_scale = np.zeros((B, Hkv, ns, d // 32), np.float32)
        self.sink_len = np.zeros(B, np.int32)
        self.ring_start = np.zeros(B, np.int32)
        self.ring_len = np.zeros(B, np.int32)
        self.seq_len = np.zeros(B, np.int32)

    def copy(self) -> "Cache":
        c = Cache.__new__(Cache)
        c.__dict__.update({k: (v.copy() if isinstance(v, np.ndarray) else v)
                           for k, v in self.__dict__.items()})
        return c


def kv_append(cache: Cache, k_new, v_new, to_sink: bool = False) -> int:
    """Quantise one token per sequence and write it into the cache in place
    (ring slot (ring_start+ring_len) mod W, or the oldest when full; or the
    next sink slot).  k_new/v_new fp32 [B][Hkv][d].  Returns rejected sink
    appends."""
    kn = _c(k_new, np.float32)
    vn = _c(v_new, np.float32)
    c = cache
    return int(_load().ndo_kv_append(
        c.B, c.Hkv, c.d, c.sink_cap, c.ring_cap, _ptr(c.k_codes), _ptr(c.k_scale),
        _ptr(c.v_codes), _ptr(c.v_scale), _ptr(c.sink_len), _ptr(c.ring_start),
        _ptr(c.ring_len), _ptr(c.seq_len), _ptr(kn), _ptr(vn), 1 if to_sink else 0))


def slot_positions(cache: Cache, b: int):
    """(kpos int64 [slots] with -1 for empty, is_sink bool [slots])."""
    ns = cache.sink_cap + cache.ring_cap
    kpos = np.empty(ns, np.int64)
    sink = np.empty(ns, np.uint8)
    _load().ndo_slot_positions(cache.sink_cap, cache.ring_cap, int(cache.sink_len[b]),
                               int(cache.ring_start[b]), int(cache.ring_len[b]),
                               int(cache.seq_len[b]), _ptr(kpos), _ptr(sink))
    return kpos, sink.astype(bool)


def decode(q, cache: Cache, window: int):
    """One decode step: q [B,Hq,d] at position seq_len-1 over every occupied
    slot under the decode mask.  Returns (out [B,Hq,d], lse [B,Hq])."""
    q = _c(q, np.float64)
    B, Hq, d = q.shape
    c = cache
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    _load().ndo_decode(B, Hq, c.Hkv, d, c.sink_cap, c.ring_cap, _ptr(q),
                       _ptr(_c(c.k_codes, np.int8)), _ptr(_c(c.k_scale, np.float32)),
                       _ptr(_c(c.v_codes, np.int8)), _ptr(_c(c.v_scale, np.float32)),
                       _ptr(_c(c.sink_len, np.int32)), _ptr(_c(c.ring_start, np.int32)),
                       _ptr(_c(c.ring_len, np.int32)), _ptr(_c(c.seq_len, np.int32)),
                       int(window), _ptr(out), _ptr(lse))
    return out, lse


# --------------------------------------------------------------------------
# Compressed attention helpers
# --------------------------------------------------------------------------

def pool_blocks(x, block: int) -> np.ndarray:
    """Mean of consecutive `block` positions: [B,T,H,d] -> [B,T//block,H,d]."""
    x = _c(x, np.float64)
    B, T, H, d = x.shape
    out = np.empty((B, T // block, H, d), np.float64)
    _load().ndo_pool_blocks(B, T, H, d, int(block), _ptr(x), _ptr(out))
    return out


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of [B,T,H,d] at positions pos [T]."""
    x = _c(x, np.float64)
    B, T, H, d = x.shape
    p = _c(pos, np.int64)
    assert p.shape == (T,)
    out = np.empty_like(x)
    _load().ndo_rope(B, T, H, d, _ptr(x), _ptr(p), float(theta), _ptr(out))
    return out


def compress(q, k, v, block: int, theta: float, table_len: Optional[int] = None):
    """_compress: returns (q rotated, [pooled K rotated at midpoints ; K rotated],
    [pooled V ; V]).  table_len defaults to T (the rotary table's length)."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    B, T, H, d = q.shape
    nb = T // block
    tl = T if table_len is None else int(table_len)
    q_out = np.empty_like(q)
    k_out = np.empty((B, nb + T, H, d), np.float64)
    v_out = np.empty((B, nb + T, H, d), np.float64)
    _load().ndo_compress(B, T, H, d, int(block), float(theta), tl, _ptr(q), _ptr(k),
                         _ptr(v), _ptr(q_out), _ptr(k_out), _ptr(v_out))
    return q_out, k_out, v_out


def chunk_prefill(q, k, v, cache: Cache, window: int):
    """Chunked prefill against the bounded cache: the chunk's tokens sit at
    positions p0 .. p0+Tc-1 (p0 = seq_len of each sequence) and each attends,
    under the decode mask ("256-token 滑动窗口：源码走读": causal, and a sink at
    any distance or qpos - kpos < window), to every occupied cache slot
    (dequantised: code * scale) and to the chunk's own keys.  Afterwards the
    chunk's tokens are appended to the ring, one kv_append each.
    q [B,Tc,Hq,d], k / v [B,Tc,Hkv,d] (already rotated).  Returns
    (out [B,Tc,Hq,d], lse [B,Tc,Hq], the cache after the appends)."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    B, Tc, Hq, d = q.shape
    out = np.empty((B, Tc, Hq, d))
    lse = np.empty((B, Tc, Hq))
    for b in range(B):
        kpos, is_sink = slot_positions(cache, b)
        occ = np.nonzero(kpos >= 0)[0]
        p0 = int(cache.seq_len[b])
        ck = dequant_g32(cache.k_codes[b][:, occ], cache.k_scale[b][:, occ]).transpose(1, 0, 2)
        cv = dequant_g32(cache.v_codes[b][:, occ], cache.v_scale[b][:, occ]).transpose(1, 0, 2)
        keys = np.concatenate([ck, k[b]], axis=0)[None]
        vals = np.concatenate([cv, v[b]], axis=0)[None]
        pos = np.concatenate([kpos[occ], p0 + np.arange(Tc)])
        snk = np.concatenate([is_sink[occ], np.zeros(Tc, bool)])
        mask = np.stack([decode_keep(p0 + t, pos, snk, window) for t in range(Tc)])
        o, l = attention(q[b][None], keys, vals, mask)
        out[b], lse[b] = o[0], l[0]
    new = cache.copy()
    for t in range(Tc):
        kv_append(new, k[:, t], v[:, t], False)
    return out, lse, new


def round_bf16(x) -> np.ndarray:
    """Storage rounding to bf16 (round to nearest even), returned as fp64:
    fp64 -> fp32 (numpy's rounding) -> bf16 on the bit pattern."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b + (((b >> 16) & 1) + np.uint32(0x7FFF))) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def compressed_cache(k, v, pos: int, window: int, block: int, theta: float,
                     n_pinned: int = 0, sink_cap: Optional[int] = None,
                     ring_cap: Optional[int] = None) -> Cache:
    """The int8 cache compressed attention decodes from after positions
    0..pos of k, v ([B, T, Hkv, d], before rotation), per "Compressed
    attention and the copy probe" ("Two kinds of columns", "Pool before
    rotating, not after"; priced in "So what happened ?"), in the library's
    layout:
      sink slot s < n_pinned   token s, key rotated at s (pinned prefix,
                               an exact key visible at any distance)
      sink slot n_pinned + j   block j of the positions after the prefix:
                               mean of its keys before rotation, rotated at
                               n_pinned + j*block + block//2; mean of values
      ring                     the newest non-pinned tokens, keys rotated at
                               their positions, in append order
    Every stored row is rounded to bf16 and quantised with quant_g32.
    sink_len counts the pinned tokens plus the pooled blocks visible to a
    query at pos: (j+1)*block <= pos - window + 1 - n_pinned."""
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    B, T, Hkv, d = k.shape
    n_tok = pos + 1
    n_pin = min(n_tok, n_pinned)
    n_rest = n_tok - n_pin
    n_blk = n_rest // block if n_tok > n_pinned else 0
    lim = pos - window + 1 - n_pinned
    n_vis = lim // block if lim >= block else 0
    S = sink_cap if sink_cap is not None else n_pinned + max(n_blk, 1)
    W = ring_cap if ring_cap is not None else window
    c = Cache(B, Hkv, d, S, W)
    kr = rope(k[:, :n_tok], np.arange(n_tok), theta) if theta else k[:, :n_tok]

    def put(slot, kk, vv):  # kk, vv [B, Hkv, d]
        c.k_codes[:, :, slot], c.k_scale[:, :, slot] = quant_g32(round_bf16(kk))
        c.v_codes[:, :, slot], c.v_scale[:, :, slot] = quant_g32(round_bf16(vv))

    for s_ in range(n_pin):
        put(s_, kr[:, s_], v[:, s_])
    if n_blk:
        seg_k = k[:, n_pinned:n_pinned + n_blk * block]
        seg_v = v[:, n_pinned:n_pinned + n_blk * block]
        pk = pool_blocks(seg_k, block)
        pv = pool_blocks(seg_v, block)
        if theta:
            mids = n_pinned + np.arange(n_blk) * block + block // 2
            pk = rope(pk, mids, theta)
        for j in range(n_blk):
            put(n_pinned + j, pk[:, j], pv[:, j])
    for i in range(max(0, n_rest - W), n_rest):  # ring index i holds token n_pinned + i
        put(S + i % W, kr[:, n_pinned + i], v[:, n_pinned + i])
    c.sink_len[:] = n_pin + n_vis
    c.ring_len[:] = min(n_rest, W)
    c.ring_start[:] = n_rest % W if n_rest > W else 0
    c.seq_len[:] = n_tok
    return c


def compressed_decode(q, k, v, pos: int, window: int, block: int, theta: float,
                      n_pinned: int = 0, sink_cap: Optional[int] = None,
                      ring_cap: Optional[int] = None):
    """Compressed attention for the query at position pos (q [B, Hq, d] before
    rotation) over compressed_cache(...): one softmax over the visible pooled
    blocks, the pinned tokens and the exact keys of the window.  Returns
    (out [B, Hq, d], lse [B, Hq], the cache)."""
    c = compressed_cache(k, v, pos, window, block, theta, n_pinned, sink_cap, ring_cap)
    qq = _c(q, np.float64)[:, None]
    if theta:
        qq = rope(qq, np.array([pos]), theta)
    out, lse = decode(qq[:, 0], c, window)
    return out, lse, c


# --------------------------------------------------------------------------
# KV budget window
# --------------------------------------------------------------------------

def kv_budget_window(d_model, attn_dim, num_heads, num_kv_heads, num_layers,
                     n_engram_sites, max_seq_len) -> int:
    """kv_budget_window ("Effective KV Window"); -1 for a divide by zero."""
    return int(_load().ndo_kv_budget_window(d_model, attn_dim or 0, num_heads,
                                            num_kv_heads, num_layers, n_engram_sites,
                                            max_seq_len))


def effective_kv_window(budget_window: int, kv_window: int) -> int:
    """effective_kv_window: min(budget, kv_window) if kv_window else budget."""
    return int(_load().ndo_effective_kv_window(budget_window, kv_window or 0))
