"""Float64 CPU oracle for one grouped-KV incremental decode step.

Test infrastructure only: the tests, the smoke check and the bench's CPU
baseline leg call it.  The product path (the C-ABI library and its Python
binding) never imports it, and it imports nothing from that path.
"""
from .oracle import (  # noqa: F401
    bf16_bits_to_f64,
    widen,
    kv_append,
    grouped_decode_attention,
    attention_weights,
    decode_step,
    kv_cache_elements,
    kv_cache_bytes_per_token,
    kv_cache_bytes,
    attention_multiplications,
    kv_append_multi,
    grouped_decode_attention_multi,
    decode_step_multi,
    to_storage,
    project_qkv,
    project_out,
    decode_layer,
    paged_rows,
    gather_paged,
    kv_append_paged,
    decode_step_paged,
    kv_append_paged_multi,
    decode_step_paged_multi,
)
