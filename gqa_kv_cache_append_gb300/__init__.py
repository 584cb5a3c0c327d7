"""GB300-native grouped-KV incremental decode attention.

The computation lives in libgqa.so (C ABI in include/gqa.h, CUDA kernels for
sm_103a under csrc/).  ``binding`` is its ctypes binding, loaded on first use
of one of the names below; ``inputs`` holds the seeded synthetic workloads.
"""
_BINDING = {
    "gqa_kv_append", "gqa_decode_attn", "gqa_decode_step", "gqa_decode_attn_noalloc",
    "gqa_kv_append_multi", "gqa_decode_attn_multi", "gqa_decode_step_multi",
    "gqa_kv_append_paged", "gqa_decode_attn_paged", "gqa_decode_step_paged",
    "gqa_project_qkv", "gqa_project_out", "gqa_decode_layer", "gqa_decode_plan",
    "gqa_device_status", "gqa_selftest_wait_timeout", "gqa_version", "decode_step", "GqaError",
    "status_string",
}


def __getattr__(name):
    if name in _BINDING:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
