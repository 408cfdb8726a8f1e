"""Thin Python binding of the C-ABI library (argument marshalling only).

Every function here forwards torch tensors' device pointers to the same-named
``extern "C"`` entry point of ``libfa_decode.so`` (declared in
``include/fa_decode.h``); all arithmetic runs in the CUDA kernels.  There is
no fallback: if the library cannot be built or loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional

import torch

from . import _build

_lock = threading.Lock()
_lib = None

FA_STATUS_LEN_CLAMPED = 1
FA_STATUS_BAD_BLOCK = 2
FA_STATUS_WAIT_TIMEOUT = 4
FA_STATUS_POS_RANGE = 8
FA_STATUS_BAD_SLOT = 16


class FaDecodeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            lib = ctypes.CDLL(path)
            P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong,
                                    ctypes.c_float, ctypes.c_size_t)
            lib.fa_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, f32, P, P, i32, i32, i32,
                                      i32, P, sz, P]
            lib.fa_decode.restype = i32
            lib.fa_decode_noalloc.argtypes = [P, P, P, P, P, P, i32, i32, i32, f32, P, P, i32,
                                              i32, i32, i32, P]
            lib.fa_decode_noalloc.restype = i32
            lib.fa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
            lib.fa_decode_workspace_size.restype = sz
            lib.fa_quantize_v_int8.argtypes = [P, i64, i32, P, P, P]
            lib.fa_quantize_v_int8.restype = i32
            lib.fa_decode_batch_invariant.argtypes = [P, P, P, P, P, P, i32, i32, i32, f32, P,
                                                      P, i32, i32, i32, i32, i32, P, sz, P]
            lib.fa_decode_batch_invariant.restype = i32
            lib.fa_decode_batch_invariant_workspace_size.argtypes = [i32, i32, i32, i32, i32,
                                                                     i32]
            lib.fa_decode_batch_invariant_workspace_size.restype = sz
            lib.fa_decode_multi_batch_invariant.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32,
                                                            f32, P, P, i32, i32, i32, i32, i32, P,
                                                            sz, P]
            lib.fa_decode_multi_batch_invariant.restype = i32
            lib.fa_decode_multi_batch_invariant_workspace_size.argtypes = [i32] * 7
            lib.fa_decode_multi_batch_invariant_workspace_size.restype = sz
            lib.fa_decode_ring_batch_invariant.argtypes = [P, P, P, P, P, i32, i32, i32, f32, P,
                                                           P, i32, i32, i32, P, sz, P]
            lib.fa_decode_ring_batch_invariant.restype = i32
            lib.fa_decode_multi.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f32, P, P, i32,
                                            i32, i32, i32, P, sz, P]
            lib.fa_decode_multi.restype = i32
            lib.fa_decode_multi_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            lib.fa_decode_multi_workspace_size.restype = sz
            lib.fa_decode_ring.argtypes = [P, P, P, P, P, i32, i32, i32, f32, P, P, i32, i32, P,
                                           sz, P]
            lib.fa_decode_ring.restype = i32
            lib.fa_append_kv_ring.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P]
            lib.fa_append_kv_ring.restype = i32
            lib.fa_decode_slots.argtypes = [P, P, P, P, P, P, i32, i32, i32, f32, P, P, i32, i32,
                                            i32, i32, P, sz, P]
            lib.fa_decode_slots.restype = i32
            lib.fa_append_kv_slots.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                               P]
            lib.fa_append_kv_slots.restype = i32
            lib.fa_append_kv.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
            lib.fa_append_kv.restype = i32
            lib.fa_gather_kv_debug.argtypes = [P, i32, P, i32, i32, i32, i32, i32, i32, P, P]
            lib.fa_gather_kv_debug.restype = i32
            lib.fa_decode_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), P]
            lib.fa_decode_device_status.restype = i32
            lib.fa_decode_profile_next.argtypes = [P, P]
            lib.fa_decode_profile_next.restype = i32
            lib.fa_selftest_wait_timeout.argtypes = [P]
            lib.fa_selftest_wait_timeout.restype = i32
            lib.fa_decode_last_error.argtypes = []
            lib.fa_decode_last_error.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("fa_decode takes device tensors")
    if not t.is_contiguous():
        raise ValueError("fa_decode takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int):
    if rc != 0:
        raise FaDecodeError(rc, load().fa_decode_last_error().decode())


def fa_decode_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                             max_kv_len: int, num_sms: int = 0) -> int:
    return int(load().fa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                               max_kv_len, num_sms))


def fa_decode(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads, n_kv_heads,
              head_dim, scale, window, out, *, batch=None, page_size=16,
              max_blocks_per_seq=None, num_blocks=None, workspace=None, stream=None):
    """One decode step: out[b,h] = softmax(scale q.K^T) V over the attended range.

    Layouts and rules are those of ``fa_decode`` in include/fa_decode.h.
    `batch` defaults to q.shape[0]; `max_blocks_per_seq` to the block table's
    row length (paged) or k_cache.shape[2] (contiguous); `num_blocks` to
    k_cache.shape[0] (paged).
    """
    if batch is None:
        batch = q.shape[0]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = block_table.shape[1] if block_table is not None else k_cache.shape[2]
    if num_blocks is None:
        num_blocks = k_cache.shape[0] if block_table is not None else 0
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales),
                          _ptr(block_table), _ptr(seq_lens), int(n_q_heads), int(n_kv_heads),
                          int(head_dim), float(scale), _ptr(window), _ptr(out), int(batch),
                          int(page_size), int(max_blocks_per_seq), int(num_blocks),
                          _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_decode_batch_invariant(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                              n_kv_heads, head_dim, scale, window, out, *, split_tokens=512,
                              batch=None, page_size=16, max_blocks_per_seq=None, num_blocks=None,
                              workspace=None, stream=None):
    """fa_decode with splits of `split_tokens` keys fixed per sequence, so a
    sequence's output is the same bytes whatever else is in the batch.
    Arguments as ``fa_decode``; the workspace is sized by
    ``fa_decode_batch_invariant_workspace_size``."""
    if batch is None:
        batch = q.shape[0]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = block_table.shape[1] if block_table is not None else k_cache.shape[2]
    if num_blocks is None:
        num_blocks = k_cache.shape[0] if block_table is not None else 0
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode_batch_invariant(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales), _ptr(block_table),
        _ptr(seq_lens), int(n_q_heads), int(n_kv_heads), int(head_dim), float(scale),
        _ptr(window), _ptr(out), int(batch), int(page_size), int(max_blocks_per_seq),
        int(num_blocks), int(split_tokens), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_decode_batch_invariant_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, max_kv_len,
                                             split_tokens=512) -> int:
    return int(load().fa_decode_batch_invariant_workspace_size(
        batch, n_q_heads, n_kv_heads, head_dim, max_kv_len, split_tokens))


def fa_decode_multi_batch_invariant(q, k_cache, v_cache, v_scales, block_table, seq_lens,
                                    n_q_heads, n_kv_heads, head_dim, scale, window, out, *,
                                    split_tokens=512, page_size=16, max_blocks_per_seq=None,
                                    num_blocks=None, workspace=None, stream=None):
    """fa_decode_multi with the batch-invariant plan (fixed splits per sequence)."""
    batch, tq = q.shape[0], q.shape[1]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = block_table.shape[1] if block_table is not None else k_cache.shape[2]
    if num_blocks is None:
        num_blocks = k_cache.shape[0] if block_table is not None else 0
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode_multi_batch_invariant(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales), _ptr(block_table),
        _ptr(seq_lens), int(tq), int(n_q_heads), int(n_kv_heads), int(head_dim), float(scale),
        _ptr(window), _ptr(out), int(batch), int(page_size), int(max_blocks_per_seq),
        int(num_blocks), int(split_tokens), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_decode_multi_batch_invariant_workspace_size(batch, n_queries, n_q_heads, n_kv_heads,
                                                   head_dim, max_kv_len, split_tokens=512) -> int:
    return int(load().fa_decode_multi_batch_invariant_workspace_size(
        batch, n_queries, n_q_heads, n_kv_heads, head_dim, max_kv_len, split_tokens))


def fa_decode_ring_batch_invariant(q, k_cache, v_cache, v_scales, seq_lens, n_q_heads,
                                   n_kv_heads, head_dim, scale, window, out, *, split_tokens=512,
                                   workspace=None, stream=None):
    """fa_decode_ring with the batch-invariant plan (fixed splits per sequence)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode_ring_batch_invariant(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales), _ptr(seq_lens), int(n_q_heads),
        int(n_kv_heads), int(head_dim), float(scale), _ptr(window), _ptr(out), int(q.shape[0]),
        int(k_cache.shape[2]), int(split_tokens), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_decode_multi(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads, n_kv_heads,
                    head_dim, scale, window, out, *, page_size=16, max_blocks_per_seq=None,
                    num_blocks=None, workspace=None, stream=None):
    """Multi-query decode: q [B, Tq, Hq, D] = each sequence's last Tq tokens,
    query j attending keys up to its own position; out [B, Tq, Hq, D]."""
    batch, tq = q.shape[0], q.shape[1]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = block_table.shape[1] if block_table is not None else k_cache.shape[2]
    if num_blocks is None:
        num_blocks = k_cache.shape[0] if block_table is not None else 0
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales),
                                _ptr(block_table), _ptr(seq_lens), int(tq), int(n_q_heads),
                                int(n_kv_heads), int(head_dim), float(scale), _ptr(window),
                                _ptr(out), int(batch), int(page_size), int(max_blocks_per_seq),
                                int(num_blocks), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_decode_multi_workspace_size(batch, n_queries, n_q_heads, n_kv_heads, head_dim, max_kv_len,
                                   num_sms=0) -> int:
    return int(load().fa_decode_multi_workspace_size(batch, n_queries, n_q_heads, n_kv_heads,
                                                     head_dim, max_kv_len, num_sms))


def fa_decode_ring(q, k_cache, v_cache, v_scales, seq_lens, n_q_heads, n_kv_heads, head_dim,
                   scale, window, out, *, workspace=None, stream=None):
    """Decode over a ring cache [B, Hkv, capacity, D]: token t at row t % capacity,
    seq_lens = tokens seen (may exceed capacity)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode_ring(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales),
                               _ptr(seq_lens), int(n_q_heads), int(n_kv_heads), int(head_dim),
                               float(scale), _ptr(window), _ptr(out), int(q.shape[0]),
                               int(k_cache.shape[2]), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_append_kv_ring(k_new, v_new, k_cache, v_cache, v_scales, positions, *, stream=None):
    """Write this step's K / V rows into a ring cache at row position % capacity."""
    rc = load().fa_append_kv_ring(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(v_scales), _ptr(positions), int(k_new.shape[0]),
                                  int(k_new.shape[1]), int(k_new.shape[2]),
                                  int(k_cache.shape[2]), _stream(stream))
    _check(rc)


def fa_decode_slots(q, k_cache, v_cache, v_scales, slot_ids, seq_lens, n_q_heads, n_kv_heads,
                    head_dim, scale, window, out, *, ring=False, workspace=None, stream=None):
    """Decode where row b reads slot slot_ids[b] of a pool [n_slots, Hkv, capacity, D]
    of contiguous (ring=False) or ring (ring=True) caches."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fa_decode_slots(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales),
                                _ptr(slot_ids), _ptr(seq_lens), int(n_q_heads), int(n_kv_heads),
                                int(head_dim), float(scale), _ptr(window), _ptr(out),
                                int(q.shape[0]), int(k_cache.shape[0]), int(k_cache.shape[2]),
                                int(bool(ring)), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def fa_append_kv_slots(k_new, v_new, k_cache, v_cache, v_scales, slot_ids, positions, *,
                       ring=False, stream=None):
    """Write row b's K / V into slot slot_ids[b] of a pool [n_slots, Hkv, capacity, D]
    at token positions[b] (row positions[b] % capacity for a ring)."""
    rc = load().fa_append_kv_slots(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(v_scales), _ptr(slot_ids), _ptr(positions),
                                   int(k_new.shape[0]), int(k_new.shape[1]), int(k_new.shape[2]),
                                   int(k_cache.shape[0]), int(k_cache.shape[2]), int(bool(ring)),
                                   _stream(stream))
    _check(rc)


def fa_decode_noalloc(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                      n_kv_heads, head_dim, scale, window, out, *, batch=None, page_size=16,
                      max_blocks_per_seq=None, num_blocks=None, stream=None):
    """fa_decode without a workspace argument, for callers that cannot allocate.

    The scratch is a fixed array inside the library (FA_NOALLOC_SCRATCH_BYTES);
    sizes that need more raise FaDecodeError.  Calls that overlap on the GPU
    share that array and race, so keep them on one stream.
    """
    if batch is None:
        batch = q.shape[0]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = block_table.shape[1] if block_table is not None else k_cache.shape[2]
    if num_blocks is None:
        num_blocks = k_cache.shape[0] if block_table is not None else 0
    rc = load().fa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scales),
                                  _ptr(block_table), _ptr(seq_lens), int(n_q_heads),
                                  int(n_kv_heads), int(head_dim), float(scale), _ptr(window),
                                  _ptr(out), int(batch), int(page_size),
                                  int(max_blocks_per_seq), int(num_blocks), _stream(stream))
    _check(rc)


def fa_quantize_v_int8(x, codes, scales, *, stream=None):
    """Pack fp32 x [..., D] into int8 codes [..., D] and fp16 scales [..., D/32]."""
    D = x.shape[-1]
    rc = load().fa_quantize_v_int8(_ptr(x), x.numel() // D, D, _ptr(codes), _ptr(scales),
                                   _stream(stream))
    _check(rc)


def fa_append_kv(k_new, v_new, k_cache, v_cache, v_scales, block_table, positions, *,
                 n_kv_heads, head_dim, page_size=16, max_blocks_per_seq=None, num_blocks=None,
                 stream=None):
    """Write this step's K / V rows ([B, Hkv, D] fp32) into the cache at `positions`."""
    batch = k_new.shape[0]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = block_table.shape[1] if block_table is not None else k_cache.shape[2]
    if num_blocks is None:
        num_blocks = k_cache.shape[0] if block_table is not None else 0
    rc = load().fa_append_kv(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                             _ptr(v_scales), _ptr(block_table), _ptr(positions), int(batch),
                             int(n_kv_heads), int(head_dim), int(page_size),
                             int(max_blocks_per_seq), int(num_blocks), _stream(stream))
    _check(rc)


def fa_gather_kv_debug(cache, row_bytes, block_table, b, n_kv_heads, page_size,
                       max_blocks_per_seq, num_blocks, n_tokens, dense, *, stream=None):
    rc = load().fa_gather_kv_debug(_ptr(cache), int(row_bytes), _ptr(block_table), int(b),
                                   int(n_kv_heads), int(page_size), int(max_blocks_per_seq),
                                   int(num_blocks), int(n_tokens), _ptr(dense), _stream(stream))
    _check(rc)


def fa_decode_profile_next(split_start=None, split_end=None):
    """Record torch.cuda.Event objects around the next call's split kernel.

    The events must already exist on the device (torch creates them lazily at
    their first record()); a zero handle raises.
    """
    a = None if split_start is None else ctypes.c_void_p(split_start.cuda_event)
    b = None if split_end is None else ctypes.c_void_p(split_end.cuda_event)
    if (split_start is not None and not a.value) or (split_end is not None and not b.value):
        raise ValueError("fa_decode_profile_next: event not created yet (record it once first)")
    _check(load().fa_decode_profile_next(a, b))


def fa_selftest_wait_timeout(*, stream=None):
    """Launch the bounded-wait self-test (about one second; sets FA_STATUS_WAIT_TIMEOUT)."""
    _check(load().fa_selftest_wait_timeout(_stream(stream)))


def fa_decode_device_status(*, stream=None) -> int:
    v = ctypes.c_uint(0)
    _check(load().fa_decode_device_status(ctypes.byref(v), _stream(stream)))
    return int(v.value)


def alloc_workspace(batch, n_q_heads, n_kv_heads, head_dim, max_kv_len, device="cuda"):
    """Device scratch for fa_decode (torch allocation: plumbing, not compute)."""
    n = fa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, max_kv_len)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)
