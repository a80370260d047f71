"""Thin Python binding of libnd's C ABI (include/nd.h).

Argument marshalling only: shapes and dtypes are read from torch tensors, their
device pointers and the current CUDA stream are passed to the C entry points,
and a non-zero status raises NDError.  Every computation runs in the CUDA
kernels of libnd.so; there is no CPU or PyTorch fallback, and importing this
module on a machine without the built library raises.  torch is used for
device memory only (outputs and workspaces the caller did not supply).

Function names match the C ABI (nd_kv_append_quant, nd_swa_sink_decode, ...).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

ND_OK, ND_ERR_INVALID_ARG, ND_ERR_UNSUPPORTED, ND_ERR_CUDA, ND_ERR_WORKSPACE, ND_ERR_DEVICE = range(6)
ND_F32, ND_BF16 = 0, 1


class NDError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = _lib().nd_status_string(status).decode()
        extra = f" (cudaError {cuda_error})" if status == ND_ERR_CUDA else ""
        super().__init__(f"{fn} failed: {name}{extra}")


class _Cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("sink_cap", ctypes.c_int), ("ring_cap", ctypes.c_int),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("sink_len", ctypes.c_void_p), ("ring_start", ctypes.c_void_p),
                ("ring_len", ctypes.c_void_p), ("seq_len", ctypes.c_void_p)]


class _CompressedCache(ctypes.Structure):
    _fields_ = [("kv", _Cache), ("k_sum", ctypes.c_void_p), ("v_sum", ctypes.c_void_p),
                ("block", ctypes.c_int), ("n_pinned", ctypes.c_int)]


class _ModelCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("d_model", "attn_dim", "num_heads", "num_kv_heads",
                                             "num_layers", "n_engram_sites", "max_seq_len",
                                             "kv_window")]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path) or _build._stale():
            path = _build.build()  # raises if the CUDA toolkit is missing
        lib = ctypes.CDLL(path)
        P, I, S, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int64
        F = ctypes.c_float
        sig = {
            "nd_version": (ctypes.c_char_p, []),
            "nd_status_string": (ctypes.c_char_p, [I]),
            "nd_last_cuda_error": (I, []),
            "nd_device_errors": (I, [P, I]),
            "nd_set_prefill_epilogue_wait_limit": (I, [ctypes.c_uint]),
            "nd_kv_append_quant": (I, [P, P, P, I, P]),
            "nd_kv_quant_rows": (I, [P, L, I, P, P, P]),
            "nd_kv_cache_from_prefill_workspace_size": (S, [I, I, I]),
            "nd_kv_cache_from_prefill": (I, [P, P, P, I, I, P, P, P, P, P, S, P]),
            "nd_swa_sink_decode_workspace_size": (S, [I, I, I, I, I]),
            "nd_swa_sink_decode": (I, [P, P, I, I, P, P, P, S, P]),
            "nd_swa_sink_decode_noalloc": (I, [P, P, I, I, P, P, P]),
            "nd_swa_sink_decode_step": (I, [P, P, P, P, I, I, P, P, P, S, P]),
            "nd_swa_sink_decode_step_host_workspace_size": (S, [I, I, I, I, I]),
            "nd_swa_sink_decode_step_host": (I, [P, P, P, P, I, I, P, P, P, S, P]),
            "nd_swa_sink_decode_step_host_packed": (I, [P, P, I, I, P, I, P, S, P]),
            "nd_compressed_decode_step_workspace_size": (S, [I, I, I, I, I]),
            "nd_compressed_decode_step": (I, [P, P, P, P, I, I, F, P, P, P, S, P]),
            "nd_swa_sink_prefill_workspace_size": (S, [I, I, I, I, I, I, F, I]),
            "nd_swa_sink_prefill": (I, [P, P, P, I, I, I, I, I, I, P, P, I, F, P, P, I, P, P, P, S, P]),
            "nd_swa_sink_prefill_tiles": (I, [P, I, I, I, I, I, F, I, P]),
            "nd_compressed_prefill_workspace_size": (S, [I, I, I, I, I, F, I]),
            "nd_compressed_prefill": (I, [P, P, P, I, I, I, I, I, I, I, I, F, P, P, P, S, P]),
            "nd_swa_sink_chunk_prefill_workspace_size": (S, [I, I, I, I, I, I, I, I]),
            "nd_swa_sink_chunk_prefill": (I, [P, P, P, I, P, I, I, P, P, P, S, P]),
            "nd_swa_sink_chunk_prefill_tiles": (I, [P, I, I, I, I, I, I, I, I, P]),
            "nd_rope_apply": (I, [P, P, I, I, I, I, F, P]),
            "nd_kv_compress_pool": (I, [P, P, I, I, I, I, I, F, P, P, P]),
            "nd_kv_compress_pool_rope_workspace_size": (S, [I, I, F]),
            "nd_kv_compress_pool_rope": (I, [P, P, I, I, I, I, I, F, P, P, P, P, S, P]),
            "nd_kv_budget_window": (I, [P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def library_path() -> str:
    _lib()
    return _build.LIB


EXPORTED = ("nd_version", "nd_status_string", "nd_last_cuda_error", "nd_device_errors",
            "nd_set_prefill_epilogue_wait_limit",
            "nd_kv_append_quant", "nd_kv_quant_rows", "nd_kv_cache_from_prefill_workspace_size", "nd_kv_cache_from_prefill", "nd_swa_sink_decode_workspace_size",
            "nd_swa_sink_decode", "nd_swa_sink_decode_noalloc", "nd_swa_sink_decode_step",
            "nd_swa_sink_decode_step_host_workspace_size", "nd_swa_sink_decode_step_host",
            "nd_swa_sink_decode_step_host_packed",
            "nd_compressed_decode_step_workspace_size", "nd_compressed_decode_step",
            "nd_swa_sink_prefill_workspace_size",
            "nd_swa_sink_prefill", "nd_swa_sink_prefill_tiles",
            "nd_compressed_prefill_workspace_size", "nd_compressed_prefill",
            "nd_swa_sink_chunk_prefill_workspace_size", "nd_swa_sink_chunk_prefill",
            "nd_swa_sink_chunk_prefill_tiles",
            "nd_rope_apply", "nd_kv_compress_pool", "nd_kv_compress_pool_rope_workspace_size",
            "nd_kv_compress_pool_rope", "nd_kv_budget_window")


def _check(fn: str, status: int):
    if status != ND_OK:
        raise NDError(fn, status, _lib().nd_last_cuda_error())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libnd takes CUDA tensors (device pointers)")
    if not t.is_contiguous():
        raise ValueError("libnd takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ND_F32
    if t.dtype == torch.bfloat16:
        return ND_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


# --------------------------------------------------------------------------
# Cache
# --------------------------------------------------------------------------

@dataclass
class KVCache:
    """Device tensors of one bounded cache in the nd_kv_cache layout."""
    k_codes: torch.Tensor   # int8 [B, Hkv, S+W, d]
    v_codes: torch.Tensor
    k_scale: torch.Tensor   # fp32 [B, Hkv, S+W, d/32]
    v_scale: torch.Tensor
    sink_len: torch.Tensor  # int32 [B]
    ring_start: torch.Tensor
    ring_len: torch.Tensor
    seq_len: torch.Tensor
    sink_cap: int
    ring_cap: int

    @classmethod
    def empty(cls, batch, n_kv_heads, head_dim, sink_cap, ring_cap, device="cuda"):
        ns = sink_cap + ring_cap
        z8 = lambda: torch.zeros((batch, n_kv_heads, ns, head_dim), dtype=torch.int8, device=device)
        zs = lambda: torch.zeros((batch, n_kv_heads, ns, head_dim // 32), dtype=torch.float32, device=device)
        zi = lambda: torch.zeros(batch, dtype=torch.int32, device=device)
        return cls(z8(), z8(), zs(), zs(), zi(), zi(), zi(), zi(), sink_cap, ring_cap)

    @property
    def batch(self):
        return self.k_codes.shape[0]

    @property
    def n_kv_heads(self):
        return self.k_codes.shape[1]

    @property
    def head_dim(self):
        return self.k_codes.shape[3]

    def struct(self) -> _Cache:
        return _Cache(self.batch, self.n_kv_heads, self.head_dim, self.sink_cap, self.ring_cap,
                      *(t.data_ptr() for t in (self.k_codes, self.v_codes, self.k_scale, self.v_scale,
                                               self.sink_len, self.ring_start, self.ring_len,
                                               self.seq_len)))


@dataclass
class CompressedCache:
    """A compressed-attention cache (nd_compressed_cache): kv's sink region
    holds n_pinned pinned tokens then the pooled blocks, its ring the exact
    window; k_sum / v_sum fp32 [B, Hkv, d] hold the open block's sums."""
    kv: KVCache
    k_sum: torch.Tensor
    v_sum: torch.Tensor
    block: int
    n_pinned: int = 0

    @classmethod
    def empty(cls, batch, n_kv_heads, head_dim, max_blocks, ring_cap, block, n_pinned=0, device="cuda"):
        kv = KVCache.empty(batch, n_kv_heads, head_dim, n_pinned + max_blocks, ring_cap, device)
        z = lambda: torch.zeros((batch, n_kv_heads, head_dim), dtype=torch.float32, device=device)
        return cls(kv, z(), z(), block, n_pinned)

    def struct(self) -> _CompressedCache:
        return _CompressedCache(self.kv.struct(), self.k_sum.data_ptr(), self.v_sum.data_ptr(), self.block,
                                self.n_pinned)


# --------------------------------------------------------------------------
# Entry points
# --------------------------------------------------------------------------

def nd_version() -> str:
    return _lib().nd_version().decode()


def nd_status_string(status: int) -> str:
    return _lib().nd_status_string(status).decode()


def nd_last_cuda_error() -> int:
    return int(_lib().nd_last_cuda_error())


def nd_device_errors(clear: bool = True) -> int:
    flags = ctypes.c_int(0)
    _check("nd_device_errors", _lib().nd_device_errors(ctypes.byref(flags), 1 if clear else 0))
    return flags.value


def nd_set_prefill_epilogue_wait_limit(polls: int) -> None:
    """Test hook: poll limit of the bf16 prefill's epilogue wait (0 = default)."""
    _check("nd_set_prefill_epilogue_wait_limit", _lib().nd_set_prefill_epilogue_wait_limit(int(polls)))


def nd_kv_append_quant(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                       to_sink: bool = False, stream=None) -> None:
    s = cache.struct()
    _check("nd_kv_append_quant", _lib().nd_kv_append_quant(
        ctypes.byref(s), _ptr(k_new), _ptr(v_new), 1 if to_sink else 0, _stream(stream)))


def nd_kv_quant_rows(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    d = x.shape[-1]
    n = x.numel() // d if d else 0
    _check("nd_kv_quant_rows", _lib().nd_kv_quant_rows(_ptr(x), n, d, _ptr(codes), _ptr(scales),
                                                       _stream(stream)))


def nd_kv_cache_from_prefill_workspace_size(cache_batch: int, sink_cap: int, ring_cap: int) -> int:
    return int(_lib().nd_kv_cache_from_prefill_workspace_size(cache_batch, sink_cap, ring_cap))


def nd_kv_cache_from_prefill(cache: KVCache, k: torch.Tensor, v: torch.Tensor, src_row: torch.Tensor,
                             seg_ids: Optional[torch.Tensor] = None, sink: Optional[torch.Tensor] = None,
                             src_seg: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                             stream=None) -> None:
    """Fill cache row e from segment src_seg[e] of batch row src_row[e] of a
    prefill's k / v (bf16 [B, T, Hkv, d]) as appending its tokens in order
    would; src_row / src_seg int32 [cache.batch] on the device."""
    B, T = k.shape[:2]
    if workspace is None:
        nbytes = nd_kv_cache_from_prefill_workspace_size(cache.batch, cache.sink_cap, cache.ring_cap)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=cache.k_codes.device)
    s = cache.struct()
    _check("nd_kv_cache_from_prefill", _lib().nd_kv_cache_from_prefill(
        ctypes.byref(s), _ptr(k), _ptr(v), B, T, _ptr(seg_ids), _ptr(sink), _ptr(src_row), _ptr(src_seg),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def nd_swa_sink_decode_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                                      max_slots: int) -> int:
    return int(_lib().nd_swa_sink_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, max_slots))


def nd_swa_sink_decode(q: torch.Tensor, cache: KVCache, window: int, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        max_slots = cache.sink_cap + cache.ring_cap
        nbytes = nd_swa_sink_decode_workspace_size(B, Hq, cache.n_kv_heads, d, max_slots)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    s = cache.struct()
    _check("nd_swa_sink_decode", _lib().nd_swa_sink_decode(
        _ptr(q), ctypes.byref(s), Hq, int(window), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out


def nd_swa_sink_decode_step(q: torch.Tensor, cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                            window: int, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Ring-append the current token (k_new, v_new: bf16 [B][Hkv][d]) and
    attend with it: nd_kv_append_quant(to_sink=False) + nd_swa_sink_decode,
    in one launch when the sequence's CTAs fit a thread-block cluster."""
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = nd_swa_sink_decode_workspace_size(B, Hq, cache.n_kv_heads, d, cache.sink_cap + cache.ring_cap)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    s = cache.struct()
    _check("nd_swa_sink_decode_step", _lib().nd_swa_sink_decode_step(
        _ptr(q), ctypes.byref(s), _ptr(k_new), _ptr(v_new), Hq, int(window), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def nd_swa_sink_decode_step_host_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                                                max_slots: int) -> int:
    return int(_lib().nd_swa_sink_decode_step_host_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                                                  max_slots))


def nd_swa_sink_decode_step_host(q_host: torch.Tensor, cache: KVCache, k_new_host: torch.Tensor,
                                 v_new_host: torch.Tensor, window: int, out_host: torch.Tensor,
                                 lse_host: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                                 stream=None, cache_struct=None) -> torch.Tensor:
    """nd_swa_sink_decode_step with q / k_new / v_new / out (/ lse) in host
    memory (CPU tensors, page-locked for asynchronous copies): the copies and
    the step are enqueued on the stream; out_host is valid once the stream
    has passed the call.  cache_struct: cache.struct(), built once by a
    caller that repeats the call on the same cache."""
    for t, name in ((q_host, "q_host"), (k_new_host, "k_new_host"), (v_new_host, "v_new_host"),
                    (out_host, "out_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    B, Hq, d = q_host.shape
    nk = cache.batch * cache.n_kv_heads * cache.head_dim
    if (B, d) != (cache.batch, cache.head_dim) or k_new_host.numel() != nk or v_new_host.numel() != nk or \
            out_host.numel() != q_host.numel() or (lse_host is not None and lse_host.numel() != B * Hq):
        raise ValueError("host buffer shapes do not match the cache")
    if workspace is None:
        nbytes = nd_swa_sink_decode_step_host_workspace_size(B, Hq, cache.n_kv_heads, d,
                                                             cache.sink_cap + cache.ring_cap)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=cache.k_codes.device)
    s = cache_struct if cache_struct is not None else cache.struct()
    _check("nd_swa_sink_decode_step_host", _lib().nd_swa_sink_decode_step_host(
        q_host.data_ptr(), ctypes.byref(s), k_new_host.data_ptr(), v_new_host.data_ptr(), Hq, int(window),
        out_host.data_ptr(), None if lse_host is None else lse_host.data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream(stream)))
    return out_host


def nd_swa_sink_decode_step_host_packed(in_host: torch.Tensor, cache: KVCache, n_q_heads: int, window: int,
                                        out_host: torch.Tensor, with_lse: bool = False,
                                        workspace: Optional[torch.Tensor] = None, stream=None,
                                        cache_struct=None) -> torch.Tensor:
    """nd_swa_sink_decode_step_host with packed host buffers: in_host one
    contiguous host tensor holding q | k_new | v_new (bf16, back to back),
    out_host one contiguous host tensor holding out (bf16) followed, with
    with_lse, by lse (fp32).  One copy each way.  Returns out_host."""
    s = cache_struct if cache_struct is not None else cache.struct()
    B, Hkv, d = s.batch, s.n_kv_heads, s.head_dim
    nin = (B * n_q_heads * d + 2 * B * Hkv * d) * 2
    nout = B * n_q_heads * d * 2 + (B * n_q_heads * 4 if with_lse else 0)
    # (this call sits on a per-token path: one cheap check per tensor)
    if in_host.is_cuda or not in_host.is_contiguous() or in_host.nbytes < nin:
        raise ValueError(f"in_host must be a contiguous host tensor of at least {nin} bytes")
    if out_host.is_cuda or not out_host.is_contiguous() or out_host.nbytes < nout:
        raise ValueError(f"out_host must be a contiguous host tensor of at least {nout} bytes")
    if workspace is None:
        nbytes = nd_swa_sink_decode_step_host_workspace_size(B, n_q_heads, Hkv, d, s.sink_cap + s.ring_cap)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=cache.k_codes.device)
    _check("nd_swa_sink_decode_step_host_packed", _lib().nd_swa_sink_decode_step_host_packed(
        in_host.data_ptr(), ctypes.byref(s), n_q_heads, window, out_host.data_ptr(),
        1 if with_lse else 0, workspace.data_ptr(), workspace.nbytes, _stream(stream)))
    return out_host


NOALLOC_SCRATCH_BYTES = 512 << 10   # ND_NOALLOC_SCRATCH_BYTES in nd.h


def nd_swa_sink_decode_noalloc(q: torch.Tensor, cache: KVCache, window: int, out: torch.Tensor,
                               lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory).  `out` must be given:
    this entry point allocates nothing.  Calls overlapping on the GPU race."""
    B, Hq, d = q.shape
    s = cache.struct()
    _check("nd_swa_sink_decode_noalloc", _lib().nd_swa_sink_decode_noalloc(
        _ptr(q), ctypes.byref(s), Hq, int(window), _ptr(out), _ptr(lse), _stream(stream)))
    return out


def nd_compressed_decode_step_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                                             max_slots: int) -> int:
    return int(_lib().nd_compressed_decode_step_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, max_slots))


def nd_compressed_decode_step(q: torch.Tensor, cache: CompressedCache, k_new: torch.Tensor, v_new: torch.Tensor,
                              window: int, rope_theta: float = 0.0, out: Optional[torch.Tensor] = None,
                              lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                              stream=None, cache_struct=None) -> torch.Tensor:
    """Append the token at position seq_len (q, k_new, v_new before rotation)
    to the compressed cache and attend with it; returns out."""
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    kv = cache.kv
    if workspace is None:
        nbytes = nd_compressed_decode_step_workspace_size(B, Hq, kv.n_kv_heads, d, kv.sink_cap + kv.ring_cap)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    s = cache_struct if cache_struct is not None else cache.struct()
    _check("nd_compressed_decode_step", _lib().nd_compressed_decode_step(
        _ptr(q), ctypes.byref(s), _ptr(k_new), _ptr(v_new), Hq, int(window), float(rope_theta), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def nd_swa_sink_prefill_workspace_size(dtype: int, batch: int, T: int, n_q_heads: int, n_kv_heads: int,
                                       head_dim: int, rope_theta: float = 0.0, block: int = 0) -> int:
    return int(_lib().nd_swa_sink_prefill_workspace_size(dtype, batch, T, n_q_heads, n_kv_heads, head_dim,
                                                         float(rope_theta), int(block)))


def nd_swa_sink_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        seg_ids: Optional[torch.Tensor] = None, sink: Optional[torch.Tensor] = None,
                        window: int = 0, rope_theta: float = 0.0,
                        pooled_k: Optional[torch.Tensor] = None, pooled_v: Optional[torch.Tensor] = None,
                        block: int = 0, out: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = nd_swa_sink_prefill_workspace_size(dt, B, T, Hq, Hkv, d, rope_theta, block)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _check("nd_swa_sink_prefill", _lib().nd_swa_sink_prefill(
        _ptr(q), _ptr(k), _ptr(v), dt, B, T, Hq, Hkv, d, _ptr(seg_ids), _ptr(sink), int(window),
        float(rope_theta), _ptr(pooled_k), _ptr(pooled_v), int(block), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def nd_swa_sink_prefill_tiles(workspace: torch.Tensor, batch: int, T: int, n_q_heads: int, n_kv_heads: int,
                              head_dim: int, rope_theta: float = 0.0, block: int = 0) -> int:
    """128-row x 64-key tile products the bf16 prefill's attention kernel
    performed in its last call on `workspace` (reads the plan; synchronises)."""
    n = ctypes.c_longlong(0)
    _check("nd_swa_sink_prefill_tiles", _lib().nd_swa_sink_prefill_tiles(
        _ptr(workspace), batch, T, n_q_heads, n_kv_heads, head_dim, float(rope_theta), int(block), ctypes.byref(n)))
    return n.value


def nd_compressed_prefill_workspace_size(batch: int, T: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                                         rope_theta: float, block: int) -> int:
    return int(_lib().nd_compressed_prefill_workspace_size(batch, T, n_q_heads, n_kv_heads, head_dim,
                                                           float(rope_theta), int(block)))


def nd_compressed_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int, block: int,
                          n_pinned: int = 0, rope_theta: float = 0.0, out: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """Compressed attention with a pinned prefix of n_pinned exact keys (bf16
    q [B, T, Hq, d], k / v [B, T, Hkv, d] before rotation); returns out."""
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = nd_compressed_prefill_workspace_size(B, T, Hq, Hkv, d, rope_theta, block)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _check("nd_compressed_prefill", _lib().nd_compressed_prefill(
        _ptr(q), _ptr(k), _ptr(v), B, T, Hq, Hkv, d, int(window), int(block), int(n_pinned), float(rope_theta),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def nd_swa_sink_chunk_prefill_workspace_size(batch: int, chunk: int, n_q_heads: int, n_kv_heads: int,
                                             head_dim: int, sink_cap: int, ring_cap: int, window: int) -> int:
    return int(_lib().nd_swa_sink_chunk_prefill_workspace_size(batch, chunk, n_q_heads, n_kv_heads, head_dim,
                                                               sink_cap, ring_cap, window))


def nd_swa_sink_chunk_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cache: KVCache, window: int,
                              out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Prefill a chunk (q [B, Tc, Hq, d], k / v [B, Tc, Hkv, d], bf16, rotated)
    against the cache, then ring-append the chunk to it; returns out."""
    B, Tc, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = nd_swa_sink_chunk_prefill_workspace_size(B, Tc, Hq, cache.n_kv_heads, d, cache.sink_cap,
                                                          cache.ring_cap, window)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    s = cache.struct()
    _check("nd_swa_sink_chunk_prefill", _lib().nd_swa_sink_chunk_prefill(
        _ptr(q), _ptr(k), _ptr(v), Tc, ctypes.byref(s), Hq, int(window), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out


def nd_swa_sink_chunk_prefill_tiles(workspace: torch.Tensor, batch: int, chunk: int, n_q_heads: int,
                                    n_kv_heads: int, head_dim: int, sink_cap: int, ring_cap: int,
                                    window: int) -> int:
    n = ctypes.c_longlong(0)
    _check("nd_swa_sink_chunk_prefill_tiles", _lib().nd_swa_sink_chunk_prefill_tiles(
        _ptr(workspace), batch, chunk, n_q_heads, n_kv_heads, head_dim, sink_cap, ring_cap, window, ctypes.byref(n)))
    return n.value


def nd_rope_apply(x: torch.Tensor, y: Optional[torch.Tensor] = None, rope_theta: float = 10000.0,
                  stream=None) -> torch.Tensor:
    B, T, H, d = x.shape
    if y is None:
        y = torch.empty_like(x)
    _check("nd_rope_apply", _lib().nd_rope_apply(_ptr(x), _ptr(y), B, T, H, d, float(rope_theta),
                                                 _stream(stream)))
    return y


def nd_kv_compress_pool(k: torch.Tensor, v: torch.Tensor, block: int, rope_theta: float = 0.0,
                        pooled_k: Optional[torch.Tensor] = None, pooled_v: Optional[torch.Tensor] = None,
                        stream=None):
    B, T, H, d = k.shape
    nb = T // block
    if pooled_k is None:
        pooled_k = torch.empty((B, nb, H, d), dtype=k.dtype, device=k.device)
    if pooled_v is None:
        pooled_v = torch.empty((B, nb, H, d), dtype=v.dtype, device=v.device)
    _check("nd_kv_compress_pool", _lib().nd_kv_compress_pool(
        _ptr(k), _ptr(v), B, T, H, d, int(block), float(rope_theta), _ptr(pooled_k), _ptr(pooled_v),
        _stream(stream)))
    return pooled_k, pooled_v


def nd_kv_compress_pool_rope_workspace_size(T: int, head_dim: int, rope_theta: float) -> int:
    return int(_lib().nd_kv_compress_pool_rope_workspace_size(T, head_dim, float(rope_theta)))


def nd_kv_compress_pool_rope(k: torch.Tensor, v: torch.Tensor, block: int, rope_theta: float = 0.0,
                             k_rot: Optional[torch.Tensor] = None, pooled_k: Optional[torch.Tensor] = None,
                             pooled_v: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                             stream=None):
    """One pass over K and V: K rotated at every position (k_rot) and the
    pooled blocks (as nd_kv_compress_pool).  Returns (k_rot, pooled_k, pooled_v)."""
    B, T, H, d = k.shape
    nb = T // block
    if k_rot is None and rope_theta:
        k_rot = torch.empty_like(k)
    if pooled_k is None:
        pooled_k = torch.empty((B, nb, H, d), dtype=k.dtype, device=k.device)
    if pooled_v is None:
        pooled_v = torch.empty((B, nb, H, d), dtype=v.dtype, device=v.device)
    if workspace is None:
        workspace = torch.empty(max(nd_kv_compress_pool_rope_workspace_size(T, d, rope_theta), 16),
                                dtype=torch.uint8, device=k.device)
    _check("nd_kv_compress_pool_rope", _lib().nd_kv_compress_pool_rope(
        _ptr(k), _ptr(v), B, T, H, d, int(block), float(rope_theta), _ptr(k_rot), _ptr(pooled_k), _ptr(pooled_v),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return k_rot, pooled_k, pooled_v


def nd_kv_budget_window(d_model: int, attn_dim: int, num_heads: int, num_kv_heads: int, num_layers: int,
                        n_engram_sites: int, max_seq_len: int, kv_window: int = 0):
    """Returns (budget window, effective window)."""
    cfg = _ModelCfg(d_model, attn_dim or 0, num_heads, num_kv_heads, num_layers, n_engram_sites,
                    max_seq_len, kv_window or 0)
    b, e = ctypes.c_int(0), ctypes.c_int(0)
    _check("nd_kv_budget_window", _lib().nd_kv_budget_window(ctypes.byref(cfg), ctypes.byref(b),
                                                             ctypes.byref(e)))
    return b.value, e.value
