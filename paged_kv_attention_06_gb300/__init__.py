"""Paged K/V attention for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``_build/libpagedattn.so`` (hand-written
CUDA kernels, declared in ``include/pagedattn.h``); ``binding`` is a thin
ctypes layer with the same entry-point names. Accessing any entry point loads
the library and raises ImportError if it has not been built: there is no CPU
or PyTorch fallback.
"""
_API = ("pa_append_kv", "pa_decode", "pa_prefill", "pa_attention", "pa_attention_route",
        "pa_decode_workspace_bytes", "pa_get_device_error", "status_string", "version",
        "pa_shape", "PagedAttentionError", "decode_workspace", "make_shape",
        "pa_debug_arm_wait_timeout", "pa_debug_prefill_variant", "pa_decode_noalloc",
        "pa_gather_kv", "pa_decode_dense", "KVCache", "KVCacheSnapshot",
        "pa_prefill_split", "pa_prefill_workspace_bytes", "prefill_workspace",
        "pa_append_kv_fp8", "pa_decode_fp8", "pa_prefill_fp8",
        "pa_prefill_fp8_workspace_bytes", "pa_attention_fp8")


def __getattr__(name):
    if name in _API or name.startswith("PA_"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)


__all__ = list(_API)
