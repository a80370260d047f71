"""sliding_window_kv_swa_gb300: SWA + KV-sink attention over a bounded int8
group-32 KV cache, and compressed attention, as hand-written CUDA kernels for
one GB300 (sm_103a) behind a C ABI (include/nd.h, libnd.so).

The Python names mirror the C entry points (every name in EXPORTED); see nd.py.
"""
from . import nd as _nd
from .nd import (  # noqa: F401
    CompressedCache, EXPORTED, KVCache, ND_BF16, ND_F32, NDError, library_path)

for _name in EXPORTED:
    globals()[_name] = getattr(_nd, _name)
del _name
