"""Pins for the oracle's multi-query decode: Tq = 1 is the single-query decode;
query j equals a single-query decode of the sequence cut after its own
position; tiny cases against an explicit causal-masked matrix product."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from test_oracle_pins import f16, make_table, scatter_pages


def _case(rng, B, Tq, Hq, Hkv, D, cap):
    q = f16(rng.standard_normal((B, Tq, Hq, D)))
    k = f16(rng.standard_normal((B, Hkv, cap, D)))
    v = f16(rng.standard_normal((B, Hkv, cap, D)))
    return q, k, v


def test_single_query_is_decode():
    rng = np.random.default_rng(51)
    q, k, v = _case(rng, 3, 1, 4, 2, 32, 40)
    lens = [40, 7, 1]
    got = oracle.decode_multi(q, k, v, lens, scale=0.3, n_kv_heads=2, window=[0, 3, 0])
    want = oracle.decode(np.ascontiguousarray(q[:, 0]), k, v, lens, scale=0.3, n_kv_heads=2,
                         window=[0, 3, 0])
    np.testing.assert_array_equal(got[:, 0], want)


@pytest.mark.parametrize("window", [0, 6])
def test_query_j_is_decode_cut_at_its_position(window):
    rng = np.random.default_rng(52)
    B, Tq, Hq, Hkv, D, cap = 2, 5, 4, 2, 32, 48
    q, k, v = _case(rng, B, Tq, Hq, Hkv, D, cap)
    lens = [48, 20]
    got = oracle.decode_multi(q, k, v, lens, scale=0.25, n_kv_heads=Hkv, window=[window] * B)
    for j in range(Tq):
        cut = [L - Tq + j + 1 for L in lens]
        want = oracle.decode(np.ascontiguousarray(q[:, j]), k, v, cut, scale=0.25,
                             n_kv_heads=Hkv, window=[window] * B)
        np.testing.assert_array_equal(got[:, j], want)


def test_more_queries_than_keys_gives_zero_rows():
    rng = np.random.default_rng(53)
    q, k, v = _case(rng, 1, 4, 2, 1, 16, 8)
    got = oracle.decode_multi(q, k, v, [2], scale=1.0, n_kv_heads=1)
    assert np.all(got[0, :2] == 0)            # positions -2, -1: no keys
    assert np.any(got[0, 2] != 0) and np.any(got[0, 3] != 0)


@pytest.mark.parametrize("seed", range(4))
def test_tiny_causal_brute_force(seed):
    rng = np.random.default_rng(60 + seed)
    B, Tq, Hkv, G, D = 2, 3, 2, 2, 8
    Hq = Hkv * G
    L = int(rng.integers(3, 9))
    q, k, v = _case(rng, B, Tq, Hq, Hkv, D, L)
    scale = float(rng.uniform(0.1, 1.0))
    got = oracle.decode_multi(q, k, v, [L, L], scale=scale, n_kv_heads=Hkv)
    for b in range(B):
        for h in range(Hq):
            Qm = q[b, :, h].astype(np.float64)                  # [Tq, D]
            K = k[b, h // G, :L].astype(np.float64)
            V = v[b, h // G, :L].astype(np.float64)
            S = Qm @ K.T * scale                                # [Tq, L]
            pos = L - Tq + np.arange(Tq)[:, None]
            S = np.where(np.arange(L)[None, :] <= pos, S, -np.inf)
            want = softmax(S, axis=1) @ V
            np.testing.assert_allclose(got[b, :, h], want, rtol=1e-12, atol=1e-13)


def test_paged_multi_equals_contiguous():
    rng = np.random.default_rng(54)
    B, Tq, Hq, Hkv, D, P = 2, 4, 4, 2, 32, 16
    lens = [37, 64]
    q, k, v = _case(rng, B, Tq, Hq, Hkv, D, 64)
    want = oracle.decode_multi(q, k, v, lens, scale=0.2, n_kv_heads=Hkv, window=[0, 9])
    bt = make_table(lens, P, 4, rng)
    got = oracle.decode_multi(q, scatter_pages(k, lens, P, bt), scatter_pages(v, lens, P, bt),
                              lens, scale=0.2, n_kv_heads=Hkv, window=[0, 9], block_table=bt,
                              page_size=P)
    np.testing.assert_array_equal(got, want)
