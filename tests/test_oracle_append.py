"""Pins for the oracle's cache append (this step's K / V rows into the cache).

Checked against numpy's own float32 -> float16 rounding (round to nearest
even), the already-pinned int8 packer, plain numpy indexing of the paged
layout, and the decode definition on the appended cache.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from test_oracle_pins import f16, make_table, scatter_pages


def _caches(rng, B, Hkv, D, cap, P, paged, int8):
    lens = [cap] * B
    k = f16(rng.standard_normal((B, Hkv, cap, D)))
    if int8:
        v, sc = oracle.pack_v_int8(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32))
    else:
        v, sc = f16(rng.standard_normal((B, Hkv, cap, D))), None
    if not paged:
        return k, v, sc, None
    bt = make_table(lens, P, cap // P, rng)
    sp = None if sc is None else scatter_pages(sc, lens, P, bt)
    return scatter_pages(k, lens, P, bt), scatter_pages(v, lens, P, bt), sp, bt


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("int8", [False, True])
def test_append_writes_exactly_the_target_rows(paged, int8):
    rng = np.random.default_rng(31)
    B, Hkv, D, cap, P = 3, 2, 64, 48, 16
    k, v, sc, bt = _caches(rng, B, Hkv, D, cap, P, paged, int8)
    kn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    pos = [5, 47, 0]
    k2, v2, sc2 = oracle.append_kv(kn, vn, k, v, pos, v_scales=sc, block_table=bt, page_size=P,
                                   max_blocks=(cap // P) if paged else cap)
    touched_k = np.zeros(k.shape[:-1], dtype=bool)
    for b in range(B):
        t = pos[b]
        for kv in range(Hkv):
            idx = (bt[b, t // P], kv, t % P) if paged else (b, kv, t)
            touched_k[idx] = True
            np.testing.assert_array_equal(k2[idx].view(np.uint16),
                                          kn[b, kv].astype(np.float16).view(np.uint16))
            if int8:
                c_want, s_want = oracle.pack_v_int8(vn[b, kv][None])
                np.testing.assert_array_equal(v2[idx], c_want[0])
                np.testing.assert_array_equal(sc2[idx].view(np.uint16), s_want[0].view(np.uint16))
            else:
                np.testing.assert_array_equal(v2[idx].view(np.uint16),
                                              vn[b, kv].astype(np.float16).view(np.uint16))
    # every other row is byte-identical
    np.testing.assert_array_equal(k2[~touched_k].view(np.uint16), k[~touched_k].view(np.uint16))
    np.testing.assert_array_equal(v2[~touched_k], v[~touched_k])
    if int8:
        np.testing.assert_array_equal(sc2[~touched_k].view(np.uint16),
                                      sc[~touched_k].view(np.uint16))


def test_append_out_of_range_is_a_no_op():
    rng = np.random.default_rng(32)
    B, Hkv, D, cap, P = 3, 2, 32, 32, 16
    k, v, sc, bt = _caches(rng, B, Hkv, D, cap, P, True, False)
    bt = bt.copy()
    bt[2, 1] = 10 ** 6                       # unmapped block for sequence 2's second page
    kn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    k2, v2, _ = oracle.append_kv(kn, kn, k, v, [-1, 32, 20], block_table=bt, page_size=P,
                                 max_blocks=cap // P)
    np.testing.assert_array_equal(k2.view(np.uint16), k.view(np.uint16))
    np.testing.assert_array_equal(v2.view(np.uint16), v.view(np.uint16))


def test_append_then_decode_attends_the_new_row():
    """Appending at position L and decoding L+1 keys equals softmax over the old
    keys plus the new one (explicit products)."""
    rng = np.random.default_rng(33)
    B, Hq, Hkv, D, cap = 1, 4, 2, 32, 40
    k, v, _, _ = _caches(rng, B, Hkv, D, cap, 16, False, False)
    L = 25
    kn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    k2, v2, _ = oracle.append_kv(kn, vn, k, v, [L])
    q = f16(rng.standard_normal((B, Hq, D)))
    got = oracle.decode(q, k2, v2, [L + 1], scale=0.3, n_kv_heads=Hkv)
    for h in range(Hq):
        kv = h // 2
        K = np.concatenate([k[0, kv, :L].astype(np.float64),
                            kn[0, kv].astype(np.float16).astype(np.float64)[None]])
        V = np.concatenate([v[0, kv, :L].astype(np.float64),
                            vn[0, kv].astype(np.float16).astype(np.float64)[None]])
        want = softmax(0.3 * (K @ q[0, h].astype(np.float64))) @ V
        np.testing.assert_allclose(got[0, h], want, rtol=1e-12, atol=1e-13)
