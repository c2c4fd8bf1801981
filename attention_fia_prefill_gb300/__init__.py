"""Fused inference attention for sm_103a (GB300): prefill, paged/MLA decode and
block-sparse attention behind a C ABI (include/fia.h), with this thin binding.

    fia_prefill(query, key, value, ...)  -> (attention_out, softmax_lse)
    fia_prefill_mla(query, key, value, query_rope=..., key_rope=..., ...)
    fia_prefill_paged(query, key_cache, value_cache, block_table, ...)
                                         -> (attention_out, softmax_lse)
    fia_decode(query, key, value, ...)   -> (attention_out, softmax_lse)
    bsa_forward(query, key, value, block_sparse_mask, block_shape, ...)

The library must have been built (attention_fia_prefill_gb300.build.build());
there is no CPU path.
"""
from ._binding import (FIAError, INT32_MAX, bsa_forward, fia_decode, fia_device_status, fia_prefill,  # noqa: F401
                       fia_prefill_mla, fia_prefill_paged, load_library)

__all__ = ["fia_prefill", "fia_prefill_mla", "fia_prefill_paged", "fia_decode", "bsa_forward", "fia_device_status", "FIAError",
           "load_library"]
