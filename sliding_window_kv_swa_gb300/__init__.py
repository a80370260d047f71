"""sliding_window_kv_swa_gb300: SWA + KV-sink attention over a bounded int8
group-32 KV cache, and compressed attention, as hand-written CUDA kernels for
one GB300 (sm_103a) behind a C ABI (include/nd.h, libnd.so).

The Python names mirror the C entry points; see nd.py.
"""
from .nd import (  # noqa: F401
    EXPORTED, KVCache, ND_BF16, ND_F32, NDError, library_path, nd_device_errors, nd_kv_append_quant,
    nd_kv_budget_window, nd_kv_compress_pool, nd_kv_quant_rows, nd_rope_apply, nd_status_string,
    nd_swa_sink_decode, nd_swa_sink_decode_noalloc, nd_swa_sink_decode_step, nd_swa_sink_decode_workspace_size,
    nd_swa_sink_decode_step_host, nd_swa_sink_decode_step_host_packed, nd_swa_sink_decode_step_host_workspace_size,
    nd_swa_sink_prefill,
    nd_swa_sink_prefill_workspace_size, nd_version)
