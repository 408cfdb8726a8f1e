"""fp64 CPU oracle for decode-step attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package.  The product path
(the CUDA library and its binding) never does, and shares no code with it.

The arithmetic lives in ``fa_oracle.c`` (plain C, double precision, built with
``-ffp-contract=off``).  This module compiles it with gcc on first use and
wraps it for numpy arrays.  Each function cites the passage it follows in the
C source; in short:

* ``decode`` -- ``softmax(q K^T * scale) V`` per query head over the attended
  range ``[lo, L)``, the definition that the online softmax and log-sum-exp
  merge of "flash_attn_vec_hybrid.metal" (mlx-native page) reach exactly;
* ``weights`` -- the softmax weights of one row (for invariant checks);
* ``pack_v_int8`` -- the symmetric int8 V codec with one fp16 scale per 32
  head_dim elements (dequantisation as ggml ``block_q8_0`` on the
  "dsv4_hc.metal" page; the quantiser rule is the plain symmetric reading);
* ``gather_rows`` -- bytes of one sequence's cache rows, gathered through the
  block table;
* ``append_kv`` -- this step's K / V rows written into the cache at each
  sequence's position (fp16 rounding, or the int8 codec for V);
* ``decode_multi`` -- several query tokens per sequence (speculative
  verify), each attending causally up to its own position;
* ``decode_ring`` / ``append_kv_ring`` -- the same over a ring cache (token t
  at row t % capacity, only the last `capacity` tokens attended);
* ``decode_slots`` / ``append_kv_slots`` -- row b uses cache slot
  ``slot_ids[b]`` of a pool of per-slot contiguous or ring caches (the slot
  map the batched kernels of "flash_attn_vec_hybrid.metal" read per row).

Every function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_oracle_append.py``, ``tests/test_oracle_ring.py``,
``tests/test_oracle_multi.py`` and ``tests/test_oracle_slots.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into oracle/_build/liboracle.so (gcc, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
    lib.oracle_fa_decode.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                     i32, dbl, P, i32, i32, P]
    lib.oracle_fa_decode.restype = i32
    lib.oracle_fa_weights.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                      dbl, i32, i32, P, P, P]
    lib.oracle_fa_weights.restype = i32
    lib.oracle_pack_v_int8.argtypes = [P, i64, i32, P, P]
    lib.oracle_pack_v_int8.restype = i32
    lib.oracle_gather_rows.argtypes = [P, i32, P, i32, i32, i32, i32, i32, P]
    lib.oracle_gather_rows.restype = i32
    lib.oracle_append_kv.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32]
    lib.oracle_append_kv.restype = i32
    lib.oracle_fa_decode_ring.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, dbl,
                                          P, i32, i32, P]
    lib.oracle_fa_decode_ring.restype = i32
    lib.oracle_fa_decode_multi.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                           i32, i32, dbl, P, i32, i32, P]
    lib.oracle_fa_decode_multi.restype = i32
    lib.oracle_append_kv_ring.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32]
    lib.oracle_append_kv_ring.restype = i32
    lib.oracle_fa_decode_slots.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                           i32, dbl, P, i32, i32, P]
    lib.oracle_fa_decode_slots.restype = i32
    lib.oracle_append_kv_slots.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32]
    lib.oracle_append_kv_slots.restype = i32
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = dbl
    lib.oracle_double_to_half.argtypes = [dbl]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _half_bits(a):
    """fp16 array -> its uint16 bit pattern (a view, no rounding)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 bits, got {a.dtype}")


def decode(q, k_cache, v_cache, seq_lens, *, scale, n_kv_heads, v_scales=None,
           block_table=None, window=None, page_size=16, max_blocks=None, rows=None,
           threads=0):
    """Oracle attention output, float64.

    q: [B, Hq, D] float16.  k_cache / v_cache: paged [num_blocks, Hkv, P, D]
    (block_table [B, max_blocks] int32) or contiguous [B, Hkv, cap, D].
    V is float16, or int8 with v_scales float16 [..., D/32].
    rows: optional int array of b*Hq+h row ids; returns [len(rows), D], else
    [B, Hq, D].
    """
    lib = _load()
    qb = _half_bits(q)
    B, Hq, D = qb.shape
    kb = _half_bits(k_cache)
    if v_scales is None:
        vb = _half_bits(v_cache)
        sb = None
    else:
        vb = _c(v_cache, np.int8)
        sb = _half_bits(v_scales)
    sl = _c(np.asarray(seq_lens, dtype=np.int32), np.int32)
    bt = None if block_table is None else _c(np.asarray(block_table, dtype=np.int32), np.int32)
    wn = None if window is None else _c(np.asarray(window, dtype=np.int32), np.int32)
    if max_blocks is None:
        max_blocks = bt.shape[1] if bt is not None else kb.shape[2]
    if rows is None:
        rr = None
        n = B * Hq
    else:
        rr = _c(np.asarray(rows, dtype=np.int32), np.int32)
        n = rr.size
    out = np.zeros((n, D), dtype=np.float64)
    rc = lib.oracle_fa_decode(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sb), _ptr(bt), _ptr(sl),
                              _ptr(wn), B, Hq, int(n_kv_heads), D, int(page_size),
                              int(max_blocks), float(scale), _ptr(rr), n, int(threads),
                              _ptr(out))
    if rc:
        raise OracleError(f"oracle_fa_decode returned {rc}")
    return out.reshape(B, Hq, D) if rows is None else out


def decode_multi(q, k_cache, v_cache, seq_lens, *, scale, n_kv_heads, v_scales=None,
                 block_table=None, window=None, page_size=16, max_blocks=None, threads=0):
    """Multi-query decode: q [B, Tq, Hq, D] = each sequence's last Tq tokens;
    query j attends keys up to its own position.  Returns [B, Tq, Hq, D]."""
    lib = _load()
    qb = _half_bits(q)
    B, Tq, Hq, D = qb.shape
    kb = _half_bits(k_cache)
    if v_scales is None:
        vb, sb = _half_bits(v_cache), None
    else:
        vb, sb = _c(v_cache, np.int8), _half_bits(v_scales)
    sl = _c(np.asarray(seq_lens, dtype=np.int32), np.int32)
    bt = None if block_table is None else _c(np.asarray(block_table, dtype=np.int32), np.int32)
    wn = None if window is None else _c(np.asarray(window, dtype=np.int32), np.int32)
    if max_blocks is None:
        max_blocks = bt.shape[1] if bt is not None else kb.shape[2]
    out = np.zeros((B * Tq * Hq, D), dtype=np.float64)
    rc = lib.oracle_fa_decode_multi(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sb), _ptr(bt), _ptr(sl),
                                    _ptr(wn), B, Tq, Hq, int(n_kv_heads), D, int(page_size),
                                    int(max_blocks), float(scale), None, 0, int(threads),
                                    _ptr(out))
    if rc:
        raise OracleError(f"oracle_fa_decode_multi returned {rc}")
    return out.reshape(B, Tq, Hq, D)


def decode_ring(q, k_cache, v_cache, seq_lens, *, scale, n_kv_heads, v_scales=None, window=None,
                rows=None, threads=0):
    """Oracle output for a ring cache [B, Hkv, capacity, D]: token t at row
    t % capacity, seq_lens = tokens seen (may exceed capacity)."""
    lib = _load()
    qb = _half_bits(q)
    B, Hq, D = qb.shape
    kb = _half_bits(k_cache)
    cap = kb.shape[2]
    if v_scales is None:
        vb, sb = _half_bits(v_cache), None
    else:
        vb, sb = _c(v_cache, np.int8), _half_bits(v_scales)
    sl = _c(np.asarray(seq_lens, dtype=np.int32), np.int32)
    wn = None if window is None else _c(np.asarray(window, dtype=np.int32), np.int32)
    if rows is None:
        rr, n = None, B * Hq
    else:
        rr = _c(np.asarray(rows, dtype=np.int32), np.int32)
        n = rr.size
    out = np.zeros((n, D), dtype=np.float64)
    rc = lib.oracle_fa_decode_ring(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sb), _ptr(sl), _ptr(wn), B,
                                   Hq, int(n_kv_heads), D, int(cap), float(scale), _ptr(rr), n,
                                   int(threads), _ptr(out))
    if rc:
        raise OracleError(f"oracle_fa_decode_ring returned {rc}")
    return out.reshape(B, Hq, D) if rows is None else out


def decode_slots(q, k_cache, v_cache, seq_lens, slot_ids, *, scale, n_kv_heads, v_scales=None,
                 window=None, ring=False, rows=None, threads=0):
    """Oracle output when row b uses cache slot slot_ids[b] of a pool
    [n_slots, Hkv, capacity, D] of contiguous (ring=False) or ring (ring=True)
    slots; q / seq_lens / window / the output are per row.  A slot id outside
    [0, n_slots) gives a zero row."""
    lib = _load()
    qb = _half_bits(q)
    B, Hq, D = qb.shape
    kb = _half_bits(k_cache)
    n_slots, cap = kb.shape[0], kb.shape[2]
    if v_scales is None:
        vb, sb = _half_bits(v_cache), None
    else:
        vb, sb = _c(v_cache, np.int8), _half_bits(v_scales)
    sl = _c(np.asarray(seq_lens, dtype=np.int32), np.int32)
    si = _c(np.asarray(slot_ids, dtype=np.int32), np.int32)
    wn = None if window is None else _c(np.asarray(window, dtype=np.int32), np.int32)
    if rows is None:
        rr, n = None, B * Hq
    else:
        rr = _c(np.asarray(rows, dtype=np.int32), np.int32)
        n = rr.size
    out = np.zeros((n, D), dtype=np.float64)
    rc = lib.oracle_fa_decode_slots(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sb), _ptr(si),
                                    int(n_slots), _ptr(sl), _ptr(wn), B, Hq, int(n_kv_heads), D,
                                    int(cap), int(bool(ring)), float(scale), _ptr(rr), n,
                                    int(threads), _ptr(out))
    if rc:
        raise OracleError(f"oracle_fa_decode_slots returned {rc}")
    return out.reshape(B, Hq, D) if rows is None else out


def append_kv_slots(k_new, v_new, k_cache, v_cache, slot_ids, positions, *, v_scales=None,
                    ring=False):
    """append_kv into a pool of per-slot caches [n_slots, Hkv, capacity, ...]:
    row b writes slot slot_ids[b] at positions[b] (row positions[b] % capacity
    for a ring).  Returns new (k_cache, v_cache, v_scales) arrays."""
    lib = _load()
    kn = _c(np.asarray(k_new, dtype=np.float32), np.float32)
    vn = _c(np.asarray(v_new, dtype=np.float32), np.float32)
    B, Hkv, D = kn.shape
    kc = np.array(k_cache, copy=True).view(np.uint16)
    vc = np.array(v_cache, copy=True)
    sc = None
    if v_scales is None:
        vc = vc.view(np.uint16)
    else:
        sc = np.array(v_scales, copy=True).view(np.uint16)
    si = _c(np.asarray(slot_ids, dtype=np.int32), np.int32)
    pos = _c(np.asarray(positions, dtype=np.int32), np.int32)
    rc = lib.oracle_append_kv_slots(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sc), _ptr(si),
                                    int(kc.shape[0]), _ptr(pos), B, Hkv, D, int(kc.shape[2]),
                                    int(bool(ring)))
    if rc:
        raise OracleError(f"oracle_append_kv_slots returned {rc}")
    if sc is None:
        return kc.view(np.float16), vc.view(np.float16), None
    return kc.view(np.float16), vc, sc.view(np.float16)


def append_kv_ring(k_new, v_new, k_cache, v_cache, positions, *, v_scales=None):
    """append_kv for a ring cache: token t goes to row t % capacity."""
    lib = _load()
    kn = _c(np.asarray(k_new, dtype=np.float32), np.float32)
    vn = _c(np.asarray(v_new, dtype=np.float32), np.float32)
    B, Hkv, D = kn.shape
    kc = np.array(k_cache, copy=True).view(np.uint16)
    vc = np.array(v_cache, copy=True)
    sc = None
    if v_scales is None:
        vc = vc.view(np.uint16)
    else:
        sc = np.array(v_scales, copy=True).view(np.uint16)
    pos = _c(np.asarray(positions, dtype=np.int32), np.int32)
    rc = lib.oracle_append_kv_ring(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sc), _ptr(pos), B,
                                   Hkv, D, int(kc.shape[2]))
    if rc:
        raise OracleError(f"oracle_append_kv_ring returned {rc}")
    if sc is None:
        return kc.view(np.float16), vc.view(np.float16), None
    return kc.view(np.float16), vc, sc.view(np.float16)


def weights(q, k_cache, seq_lens, b, h, *, scale, n_kv_heads, block_table=None,
            window=None, page_size=16, max_blocks=None):
    """Softmax weights of row (b, h) over its attended range: (lo, hi, p[hi-lo])."""
    lib = _load()
    qb = _half_bits(q)
    B, Hq, D = qb.shape
    kb = _half_bits(k_cache)
    sl = _c(np.asarray(seq_lens, dtype=np.int32), np.int32)
    bt = None if block_table is None else _c(np.asarray(block_table, dtype=np.int32), np.int32)
    wn = None if window is None else _c(np.asarray(window, dtype=np.int32), np.int32)
    if max_blocks is None:
        max_blocks = bt.shape[1] if bt is not None else kb.shape[2]
    p = np.zeros(max(int(sl[b]), 1), dtype=np.float64)
    lo = ctypes.c_int()
    hi = ctypes.c_int()
    rc = lib.oracle_fa_weights(_ptr(qb), _ptr(kb), _ptr(bt), _ptr(sl), _ptr(wn), B, Hq,
                               int(n_kv_heads), D, int(page_size), int(max_blocks),
                               float(scale), int(b), int(h), _ptr(p), ctypes.byref(lo),
                               ctypes.byref(hi))
    if rc:
        raise OracleError(f"oracle_fa_weights returned {rc}")
    return lo.value, hi.value, p[: hi.value - lo.value].copy()


def pack_v_int8(x):
    """Quantise fp32 rows [..., D] into (int8 codes [..., D], fp16 scales [..., D/32])."""
    lib = _load()
    x = _c(np.asarray(x, dtype=np.float32), np.float32)
    D = x.shape[-1]
    n = x.size // D
    codes = np.zeros(x.shape, dtype=np.int8)
    scales = np.zeros(x.shape[:-1] + (D // 32,), dtype=np.uint16)
    rc = lib.oracle_pack_v_int8(_ptr(x), n, D, _ptr(codes), _ptr(scales))
    if rc:
        raise OracleError(f"oracle_pack_v_int8 returned {rc}")
    return codes, scales.view(np.float16)


def gather_rows(cache, block_table, b, n_tokens, *, n_kv_heads, page_size=16,
                max_blocks=None):
    """Bytes of sequence b's first n_tokens rows, gathered: [Hkv, n_tokens, row...]."""
    lib = _load()
    cache = np.ascontiguousarray(cache)
    row_shape = cache.shape[3:]
    row_bytes = int(np.prod(row_shape)) * cache.itemsize
    bt = None if block_table is None else _c(np.asarray(block_table, dtype=np.int32), np.int32)
    if max_blocks is None:
        max_blocks = bt.shape[1] if bt is not None else cache.shape[2]
    dense = np.zeros((n_kv_heads, n_tokens) + row_shape, dtype=cache.dtype)
    rc = lib.oracle_gather_rows(_ptr(cache), row_bytes, _ptr(bt), int(b), int(n_kv_heads),
                                int(page_size), int(max_blocks), int(n_tokens), _ptr(dense))
    if rc:
        raise OracleError(f"oracle_gather_rows returned {rc}")
    return dense


def append_kv(k_new, v_new, k_cache, v_cache, positions, *, v_scales=None, block_table=None,
              page_size=16, max_blocks=None, num_blocks=None):
    """Write k_new / v_new ([B, Hkv, D] fp32) into copies of the caches at each
    sequence's position; returns (k_cache, v_cache, v_scales) as new arrays."""
    lib = _load()
    kn = _c(np.asarray(k_new, dtype=np.float32), np.float32)
    vn = _c(np.asarray(v_new, dtype=np.float32), np.float32)
    B, Hkv, D = kn.shape
    kc = np.array(k_cache, copy=True).view(np.uint16)
    vc = np.array(v_cache, copy=True)
    if v_scales is None:
        vc = vc.view(np.uint16)
        sc = None
    else:
        if vc.dtype != np.int8:
            raise TypeError("int8 V cache expected with v_scales")
        sc = np.array(v_scales, copy=True).view(np.uint16)
    pos = _c(np.asarray(positions, dtype=np.int32), np.int32)
    bt = None if block_table is None else _c(np.asarray(block_table, dtype=np.int32), np.int32)
    if max_blocks is None:
        max_blocks = bt.shape[1] if bt is not None else kc.shape[2]
    if num_blocks is None:
        num_blocks = kc.shape[0] if bt is not None else 0
    rc = lib.oracle_append_kv(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sc), _ptr(bt),
                              _ptr(pos), B, Hkv, D, int(page_size), int(max_blocks),
                              int(num_blocks))
    if rc:
        raise OracleError(f"oracle_append_kv returned {rc}")
    kc = kc.view(np.float16)
    if sc is None:
        return kc, vc.view(np.float16), None
    return kc, vc, sc.view(np.float16)


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(bits)


def double_to_half(x: float) -> int:
    return _load().oracle_double_to_half(x)
