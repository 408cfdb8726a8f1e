"""GB300 (sm_103a) decode-step attention over a paged or contiguous KV cache.

The compute lives in the CUDA library built from ``csrc/fa_decode.cu``
(C ABI in ``include/fa_decode.h``); ``binding`` forwards torch tensors to it.
``inputs`` draws the seeded synthetic workloads.
"""
from .binding import (FaDecodeError, fa_append_kv, fa_append_kv_ring, fa_decode_multi,
                      fa_decode_batch_invariant, fa_decode_batch_invariant_workspace_size,
                      fa_decode_multi_batch_invariant,
                      fa_decode_multi_batch_invariant_workspace_size,
                      fa_decode_ring_batch_invariant,
                      fa_decode_multi_workspace_size, fa_decode_ring, fa_decode_slots,
                      fa_append_kv_slots, alloc_workspace, fa_decode, fa_decode_device_status,  # noqa: F401
                      fa_decode_profile_next, fa_decode_workspace_size, fa_gather_kv_debug,
                      fa_quantize_v_int8, load)

__all__ = ["fa_decode", "fa_decode_batch_invariant", "fa_decode_batch_invariant_workspace_size",
           "fa_decode_multi_batch_invariant", "fa_decode_multi_batch_invariant_workspace_size",
           "fa_decode_ring_batch_invariant",
           "fa_decode_multi", "fa_decode_multi_workspace_size", "fa_decode_ring", "fa_decode_slots", "fa_append_kv_slots", "fa_append_kv", "fa_append_kv_ring", "fa_decode_workspace_size", "fa_quantize_v_int8", "fa_gather_kv_debug",
           "fa_decode_device_status", "fa_decode_profile_next", "alloc_workspace", "FaDecodeError", "load"]
