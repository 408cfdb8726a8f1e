"""Pins for the oracle's ring cache: a ring of capacity C holding the last C
of N tokens (token t at row t % C) equals a plain contiguous cache of those
tokens, for every window; appending into the ring writes row t % C."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import f16


def _stream(rng, B, Hkv, D, N):
    """The full token stream of each sequence (N tokens), as a contiguous cache."""
    return f16(rng.standard_normal((B, Hkv, N, D))), f16(rng.standard_normal((B, Hkv, N, D)))


def _ring_of(full, C, n_seen):
    """Ring storage of capacity C after n_seen[b] tokens of each sequence."""
    B, Hkv, N, D = full.shape
    ring = np.full((B, Hkv, C, D), np.nan, dtype=full.dtype)
    for b in range(B):
        for t in range(n_seen[b]):
            ring[b, :, t % C] = full[b, :, t]
    return ring


@pytest.mark.parametrize("window", [0, 5, 16, 40, 1000])
def test_ring_equals_contiguous_last_capacity_tokens(window):
    rng = np.random.default_rng(41)
    B, Hq, Hkv, D, C = 4, 4, 2, 32, 32
    n_seen = [7, 32, 33, 100]                     # below, at, just past and far past capacity
    K, V = _stream(rng, B, Hkv, D, max(n_seen))
    q = f16(rng.standard_normal((B, Hq, D)))
    got = oracle.decode_ring(q, _ring_of(K, C, n_seen), _ring_of(V, C, n_seen), n_seen,
                             scale=0.2, n_kv_heads=Hkv, window=[window] * B)
    for b in range(B):
        N = n_seen[b]
        lo = max(0, N - C)
        if window:
            lo = max(lo, N - window)
        want = oracle.decode(q[b:b + 1], np.ascontiguousarray(K[b:b + 1, :, lo:N]),
                             np.ascontiguousarray(V[b:b + 1, :, lo:N]), [N - lo], scale=0.2,
                             n_kv_heads=Hkv)
        np.testing.assert_array_equal(got[b], want[0])


def test_ring_below_capacity_equals_plain_contiguous():
    rng = np.random.default_rng(42)
    K, V = _stream(rng, 2, 2, 16, 20)
    q = f16(rng.standard_normal((2, 4, 16)))
    got = oracle.decode_ring(q, K, V, [20, 9], scale=0.5, n_kv_heads=2)
    want = oracle.decode(q, K, V, [20, 9], scale=0.5, n_kv_heads=2)
    np.testing.assert_array_equal(got, want)


def test_ring_int8_v_equals_contiguous():
    rng = np.random.default_rng(43)
    B, Hq, Hkv, D, C = 2, 4, 2, 64, 32
    n_seen = [50, 64]
    K, _ = _stream(rng, B, Hkv, D, 64)
    codes, sc = oracle.pack_v_int8(rng.standard_normal((B, Hkv, 64, D)).astype(np.float32))
    q = f16(rng.standard_normal((B, Hq, D)))
    ring_c = np.zeros((B, Hkv, C, D), dtype=np.int8)
    ring_s = np.zeros((B, Hkv, C, D // 32), dtype=np.float16)
    for b in range(B):
        for t in range(n_seen[b]):
            ring_c[b, :, t % C] = codes[b, :, t]
            ring_s[b, :, t % C] = sc[b, :, t]
    got = oracle.decode_ring(q, _ring_of(K, C, n_seen), ring_c, n_seen, scale=0.1, n_kv_heads=2,
                             v_scales=ring_s)
    for b in range(B):
        N = n_seen[b]
        want = oracle.decode(q[b:b + 1], np.ascontiguousarray(K[b:b + 1, :, N - C:N]),
                             np.ascontiguousarray(codes[b:b + 1, :, N - C:N]), [C], scale=0.1,
                             n_kv_heads=2, v_scales=np.ascontiguousarray(sc[b:b + 1, :, N - C:N]))
        np.testing.assert_array_equal(got[b], want[0])


def test_ring_append_writes_row_t_mod_capacity():
    rng = np.random.default_rng(44)
    B, Hkv, D, C = 3, 2, 32, 16
    k = f16(rng.standard_normal((B, Hkv, C, D)))
    v = f16(rng.standard_normal((B, Hkv, C, D)))
    kn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    pos = [3, 16, 1000]
    k2, v2, _ = oracle.append_kv_ring(kn, vn, k, v, pos)
    for b in range(B):
        r = pos[b] % C
        np.testing.assert_array_equal(k2[b, :, r].view(np.uint16),
                                      kn[b].astype(np.float16).view(np.uint16))
        np.testing.assert_array_equal(v2[b, :, r].view(np.uint16),
                                      vn[b].astype(np.float16).view(np.uint16))
        others = [i for i in range(C) if i != r]
        np.testing.assert_array_equal(k2[b, :, others].view(np.uint16),
                                      k[b, :, others].view(np.uint16))
    # a negative position writes nothing
    k3, _, _ = oracle.append_kv_ring(kn, vn, k, v, [-1, -5, -16])
    np.testing.assert_array_equal(k3.view(np.uint16), k.view(np.uint16))
