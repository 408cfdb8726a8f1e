"""Pins for the oracle's slot map: row b of a step using cache slot
slot_ids[b] of a pool equals the plain decode of the gathered sub-pool (row b
given slot slot_ids[b]'s cache as its own), bit for bit, for contiguous and
ring slots; a slot id that names no slot gives a zero row; appending through
the map writes exactly the mapped slot's row."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import f16


def _pool(rng, n_slots, Hkv, C, D):
    return (f16(rng.standard_normal((n_slots, Hkv, C, D))),
            f16(rng.standard_normal((n_slots, Hkv, C, D))))


@pytest.mark.parametrize("window", [0, 9])
def test_slot_map_equals_gathered_sub_batch(window):
    rng = np.random.default_rng(61)
    n_slots, Hq, Hkv, D, C = 9, 4, 2, 32, 48
    K, V = _pool(rng, n_slots, Hkv, C, D)
    slots = np.array([7, 2, 5, 0, 2], dtype=np.int32)     # a permuted subset, one repeated
    lens = [48, 13, 1, 30, 40]
    B = len(slots)
    q = f16(rng.standard_normal((B, Hq, D)))
    win = [window] * B
    got = oracle.decode_slots(q, K, V, lens, slots, scale=0.3, n_kv_heads=Hkv, window=win)
    want = oracle.decode(q, np.ascontiguousarray(K[slots]), np.ascontiguousarray(V[slots]), lens,
                         scale=0.3, n_kv_heads=Hkv, window=win)
    np.testing.assert_array_equal(got, want)
    # and the map matters: the gathered pool in batch order gives different rows
    plain = oracle.decode(q, np.ascontiguousarray(K[:B]), np.ascontiguousarray(V[:B]), lens,
                          scale=0.3, n_kv_heads=Hkv, window=win)
    assert not np.array_equal(got[0], plain[0])


def test_identity_map_equals_plain_decode():
    rng = np.random.default_rng(62)
    K, V = _pool(rng, 4, 2, 32, 16)
    q = f16(rng.standard_normal((4, 4, 16)))
    lens = [32, 5, 0, 17]
    got = oracle.decode_slots(q, K, V, lens, np.arange(4, dtype=np.int32), scale=0.5,
                              n_kv_heads=2)
    want = oracle.decode(q, K, V, lens, scale=0.5, n_kv_heads=2)
    np.testing.assert_array_equal(got, want)


def test_slot_out_of_range_gives_zero_row():
    rng = np.random.default_rng(63)
    K, V = _pool(rng, 3, 2, 16, 16)
    q = f16(rng.standard_normal((3, 4, 16)))
    got = oracle.decode_slots(q, K, V, [16, 16, 16], np.array([1, 3, -1], dtype=np.int32),
                              scale=0.5, n_kv_heads=2)
    assert np.all(got[1:] == 0.0)
    want = oracle.decode(q[:1], np.ascontiguousarray(K[1:2]), np.ascontiguousarray(V[1:2]), [16],
                         scale=0.5, n_kv_heads=2)
    np.testing.assert_array_equal(got[0], want[0])


@pytest.mark.parametrize("int8", [False, True])
def test_ring_slots_equal_ring_of_gathered_slots(int8):
    rng = np.random.default_rng(64 + int8)
    n_slots, Hq, Hkv, D, C = 6, 4, 2, 64, 32
    K = f16(rng.standard_normal((n_slots, Hkv, C, D)))
    if int8:
        V, S = oracle.pack_v_int8(rng.standard_normal((n_slots, Hkv, C, D)).astype(np.float32))
    else:
        V, S = f16(rng.standard_normal((n_slots, Hkv, C, D))), None
    slots = np.array([4, 1, 5], dtype=np.int32)
    seen = [7, 32, 100]                         # below, at and far past capacity
    q = f16(rng.standard_normal((3, Hq, D)))
    got = oracle.decode_slots(q, K, V, seen, slots, scale=0.2, n_kv_heads=Hkv, v_scales=S,
                              ring=True)
    want = oracle.decode_ring(q, np.ascontiguousarray(K[slots]), np.ascontiguousarray(V[slots]),
                              seen, scale=0.2, n_kv_heads=Hkv,
                              v_scales=None if S is None else np.ascontiguousarray(S[slots]))
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("ring", [False, True])
def test_append_through_slot_map_writes_the_mapped_row(ring):
    rng = np.random.default_rng(66 + ring)
    n_slots, Hkv, D, C = 5, 2, 32, 16
    K, V = _pool(rng, n_slots, Hkv, C, D)
    slots = np.array([3, 0, 7, 1], dtype=np.int32)       # 7 names no slot: nothing written
    pos = [4, 15, 2, 40 if ring else 9]
    kn = rng.standard_normal((4, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((4, Hkv, D)).astype(np.float32)
    k2, v2, _ = oracle.append_kv_slots(kn, vn, K, V, slots, pos, ring=ring)
    want_k, want_v = K.view(np.uint16).copy(), V.view(np.uint16).copy()
    for b, s in enumerate(slots):
        if s >= n_slots:
            continue
        r = pos[b] % C if ring else pos[b]
        want_k[s, :, r] = kn[b].astype(np.float16).view(np.uint16)
        want_v[s, :, r] = vn[b].astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(k2.view(np.uint16), want_k)
    np.testing.assert_array_equal(v2.view(np.uint16), want_v)


def test_append_through_slot_map_int8_equals_packer():
    rng = np.random.default_rng(68)
    n_slots, Hkv, D, C = 4, 2, 64, 16
    K = f16(rng.standard_normal((n_slots, Hkv, C, D)))
    V, S = oracle.pack_v_int8(rng.standard_normal((n_slots, Hkv, C, D)).astype(np.float32))
    slots = np.array([2, 3], dtype=np.int32)
    kn = rng.standard_normal((2, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((2, Hkv, D)).astype(np.float32)
    _, v2, s2 = oracle.append_kv_slots(kn, vn, K, V, slots, [5, 0], v_scales=S)
    codes, sc = oracle.pack_v_int8(vn)
    np.testing.assert_array_equal(v2[2, :, 5], codes[0])
    np.testing.assert_array_equal(s2[3, :, 0].view(np.uint16), sc[1].view(np.uint16))
    untouched = np.ones(v2.shape[:3], dtype=bool)
    untouched[2, :, 5] = untouched[3, :, 0] = False
    np.testing.assert_array_equal(v2[untouched], V[untouched])
