"""MQA / GQA incremental decode attention for NVIDIA B300 (sm_103a).

The compute lives in ``libmqa.so`` (hand-written CUDA behind a C ABI, declared in
``include/mqa.h``). :mod:`query_grouped_decode_kv_b300.binding` marshals torch tensors into that ABI;
it computes nothing itself. Importing a binding name loads the library and fails loudly if it has
not been built.
"""
from __future__ import annotations

_BINDING_NAMES = {
    "kv_append", "decode_attention", "decode_step", "kv_append_paged", "decode_attention_paged",
    "decode_step_paged", "kv_append_fp8", "decode_attention_fp8", "decode_step_fp8",
    "kv_append_multi", "decode_attention_multi", "decode_step_multi",
    "kv_append_paged_fp8", "decode_attention_paged_fp8", "decode_step_paged_fp8",
    "kv_append_paged_multi", "decode_attention_paged_multi", "decode_step_paged_multi",
    "get_device_status", "status_string", "MqaError", "set_launch_overlap",
    "library_path", "kernel_launch_count", "debug_override", "debug_timeout_site", "debug_set_wait_limit_ns", "debug_stall", "raw",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
