"""Pins for the fp64 CPU oracle: each check ties it to something other than itself.

Closed forms, invariants, special cases that reduce to a library routine
(scipy's softmax, numpy's mean), brute force on tiny inputs and hand-derived
golden cases (tests/golden/).  Together they catch a dropped term, a wrong
sign or index, a transposed operand, a wrong head map, an off-by-one window
or a wrong block-table index anywhere in the oracle.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(a):
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def contiguous_case(rng, B, Hq, Hkv, D, cap):
    q = f16(rng.standard_normal((B, Hq, D)))
    k = f16(rng.standard_normal((B, Hkv, cap, D)))
    v = f16(rng.standard_normal((B, Hkv, cap, D)))
    return q, k, v


def make_table(lens, P, max_blocks, rng):
    """Random-permutation block table: sequence b's page p -> a physical block."""
    nb = [-(-L // P) for L in lens]
    perm = rng.permutation(sum(nb)).astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nb):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt


def scatter_pages(cache, lens, P, bt):
    """Copy a contiguous [B,Hkv,cap,...] cache into pages [blocks,Hkv,P,...] via bt."""
    B, Hkv = cache.shape[:2]
    total = int(bt.max()) + 1
    pages = np.zeros((total, Hkv, P) + cache.shape[3:], dtype=cache.dtype)
    for b in range(B):
        for t in range(lens[b]):
            pages[bt[b, t // P], :, t % P] = cache[b, :, t]
    return pages


def to_paged(cache, lens, P, rng):
    bt = make_table(lens, P, -(-cache.shape[2] // P), rng)
    return scatter_pages(cache, lens, P, bt), bt


# ----------------------------------------------------------------- golden files

def parse_cases(path):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case "):
            cur = {"name": line[5:].strip()}
            cases.append(cur)
            continue
        key, val = (s.strip() for s in line.split("=", 1))
        cur[key] = val
    return cases


def parse_tensor(text):
    heads = [h.strip() for h in text.split("|")]
    return np.array([[[float(x) for x in row.split(",")] for row in h.split(";")]
                     for h in heads])


def parse_scale(text):
    if text.startswith("ln("):
        return math.log(float(text[3:-1]))
    return float(text)


@pytest.mark.parametrize("case", parse_cases(os.path.join(GOLDEN, "closed_form_attention.txt")),
                         ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    Hq, Hkv, D, L, W = (int(case[k]) for k in ("Hq", "Hkv", "D", "L", "W"))
    q = parse_tensor(case["q"]).reshape(1, Hq, D)
    k = parse_tensor(case["k"]).reshape(1, Hkv, -1, D)
    v = parse_tensor(case["v"]).reshape(1, Hkv, -1, D)
    want = parse_tensor(case["out"]).reshape(Hq, D)
    got = oracle.decode(f16(q), f16(k), f16(v), [L], scale=parse_scale(case["scale"]),
                        n_kv_heads=Hkv, window=[W])
    np.testing.assert_allclose(got[0], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", parse_cases(os.path.join(GOLDEN, "int8_pack_cases.txt")),
                         ids=lambda c: c["name"])
def test_golden_int8_pack(case):
    x = np.zeros((1, 32), dtype=np.float32)
    vals = [float(s) for s in case["x"].split(",")]
    x[0, :len(vals)] = vals
    want_codes = np.zeros(32, dtype=np.int8)
    cl = [int(s) for s in case["codes"].split(",")]
    want_codes[:len(cl)] = cl
    codes, scales = oracle.pack_v_int8(x)
    assert int(scales.view(np.uint16)[0, 0]) == int(case["scale_bits"], 16)
    np.testing.assert_array_equal(codes[0], want_codes)


# ----------------------------------------------------------------- fp16 codec

def test_half_decode_matches_numpy():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    finite = np.isfinite(r)
    np.testing.assert_array_equal(got[finite], r[finite])
    assert np.all(np.isnan(got[np.isnan(r)]))


def test_half_encode_round_nearest_even():
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.standard_normal(4000) * 10 ** rng.uniform(-9, 4, 4000),
                         [0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25,
                          3 * 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]])
    for x in xs:
        with np.errstate(over="ignore"):
            want = np.float16(x).view(np.uint16)  # numpy rounds to nearest even
        assert oracle.double_to_half(float(x)) == int(want), x


# ----------------------------------------------------------------- int8 packer

def test_int8_pack_error_bound_and_full_range():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    codes, scales = oracle.pack_v_int8(x)
    s = np.repeat(scales.astype(np.float64), 32, axis=1)
    deq = codes.astype(np.float64) * s
    xb = x.astype(np.float64)
    # every element within half a step (clamped extremes within half a step
    # plus the scale's own fp16 rounding, 127 * ulp(s) / 2)
    slack = s / 2 + 127 * s * 2.0 ** -11
    assert np.all(np.abs(deq - xb) <= slack)
    inner = np.abs(xb) < 126 * s
    assert np.all(np.abs(deq - xb)[inner] <= s[inner] / 2 + 1e-12)
    # the largest magnitude of each block codes to +-127
    blk = np.abs(codes.reshape(64, 8, 32).astype(np.int32)).max(-1)
    assert np.all(blk == 127)
    assert codes.min() >= -127
    # scales are the rounded amax/127
    amax = np.abs(x.reshape(64, 8, 32)).max(-1).astype(np.float64)
    np.testing.assert_array_equal(scales, (amax / 127).astype(np.float16))


def test_int8_blocks_are_independent():
    x = np.zeros((1, 64), dtype=np.float32)
    x[0, :4] = [127, -63.5, 0.5, 1.5]
    x[0, 32:35] = [1.0, 0.5, -0.25]
    codes, scales = oracle.pack_v_int8(x)
    assert list(scales.view(np.uint16)[0]) == [0x3C00, 0x2008]
    assert list(codes[0, :4]) == [127, -64, 0, 2]
    assert list(codes[0, 32:35]) == [127, 64, -32]


# ----------------------------------------------------------------- attention

def brute_force(q, k, v, scale, lo, hi):
    """Explicit matrix products for one head: softmax(q K^T * scale) V (float64)."""
    K = k[lo:hi].astype(np.float64)
    V = v[lo:hi].astype(np.float64)
    s = (K @ q.astype(np.float64)) * scale
    return softmax(s) @ V


@pytest.mark.parametrize("seed", range(6))
def test_tiny_brute_force(seed):
    rng = np.random.default_rng(seed)
    B, Hkv, G = 3, 2, 2
    Hq = Hkv * G
    D = int(rng.choice([4, 6, 8]))
    lens = [int(x) for x in rng.integers(1, 9, B)]
    cap = max(lens)
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, cap)
    scale = float(rng.uniform(0.1, 2.0))
    got = oracle.decode(q, k, v, lens, scale=scale, n_kv_heads=Hkv)
    for b in range(B):
        for h in range(Hq):
            want = brute_force(q[b, h], k[b, h // G], v[b, h // G], scale, 0, lens[b])
            np.testing.assert_allclose(got[b, h], want, rtol=1e-13, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    B, Hq, Hkv, D, L = 1, 4, 2, 16, 37
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, L)
    k[:] = k[:, :, :1, :]
    got = oracle.decode(q, k, v, [L], scale=0.7, n_kv_heads=Hkv)
    for h in range(Hq):
        want = v[0, h // 2].astype(np.float64).mean(0)
        np.testing.assert_allclose(got[0, h], want, rtol=1e-12, atol=1e-13)


def test_dominant_logit_returns_its_value_row():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, D, L, star = 1, 1, 1, 32, 50, 17
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, L)
    k[:] = 0
    k[0, 0, star] = f16(q[0, 0].astype(np.float64) * 4)
    got = oracle.decode(q, k, v, [L], scale=100.0, n_kv_heads=Hkv)
    np.testing.assert_allclose(got[0, 0], v[0, 0, star].astype(np.float64), rtol=0, atol=1e-12)


def test_weights_sum_to_one_and_order_by_score():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, L = 2, 4, 2, 64, 300
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, L)
    for b in range(B):
        for h in range(Hq):
            lo, hi, p = oracle.weights(q, k, [L, L - 40], b, h, scale=0.125, n_kv_heads=Hkv)
            assert (lo, hi) == (0, L - 40 * b)
            assert abs(p.sum() - 1.0) < 1e-14
            assert np.all(p > 0)
            scores = k[b, h // 2, lo:hi].astype(np.float64) @ q[b, h].astype(np.float64)
            assert np.argmax(p) == np.argmax(scores)
            # ratio of two weights is exp of the score difference
            i, j = 3, 200
            assert math.isclose(p[i] / p[j], math.exp(0.125 * (scores[i] - scores[j])),
                                rel_tol=1e-11)


def test_length_one_returns_first_value_exactly():
    rng = np.random.default_rng(6)
    q, k, v = contiguous_case(rng, 2, 4, 2, 128, 5)
    got = oracle.decode(q, k, v, [1, 1], scale=0.3, n_kv_heads=2)
    for b in range(2):
        for h in range(4):
            np.testing.assert_array_equal(got[b, h], v[b, h // 2, 0].astype(np.float64))


def test_zero_length_gives_zeros():
    rng = np.random.default_rng(6)
    q, k, v = contiguous_case(rng, 2, 4, 2, 32, 5)
    got = oracle.decode(q, k, v, [0, 5], scale=0.3, n_kv_heads=2)
    assert np.all(got[0] == 0)
    assert np.any(got[1] != 0)


def test_scale_zero_is_uniform_average():
    rng = np.random.default_rng(8)
    L = 123
    q, k, v = contiguous_case(rng, 1, 2, 1, 32, L)
    got = oracle.decode(q, k, v, [L], scale=0.0, n_kv_heads=1)
    want = v[0, 0].astype(np.float64).mean(0)
    for h in range(2):
        np.testing.assert_allclose(got[0, h], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("W", [1, 7, 16, 99, 200, 500])
def test_window_equals_dense_slice(W):
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D, L = 2, 4, 2, 32, 200
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, L)
    got = oracle.decode(q, k, v, [L, L], scale=0.2, n_kv_heads=Hkv, window=[W, 0])
    lo = max(0, L - W)
    ks = np.ascontiguousarray(k[:, :, lo:])
    vs = np.ascontiguousarray(v[:, :, lo:])
    want = oracle.decode(q, ks, vs, [L - lo, L - lo], scale=0.2, n_kv_heads=Hkv)
    np.testing.assert_array_equal(got[0], want[0])
    full = oracle.decode(q, k, v, [L, L], scale=0.2, n_kv_heads=Hkv)
    np.testing.assert_array_equal(got[1], full[1])


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(10)
    B, Hq, Hkv, D, L = 2, 8, 2, 32, 40
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, L)
    got = oracle.decode(q, k, v, [L, 33], scale=0.2, n_kv_heads=Hkv)
    krep = np.repeat(k, Hq // Hkv, axis=1)
    vrep = np.repeat(v, Hq // Hkv, axis=1)
    want = oracle.decode(q, krep, vrep, [L, 33], scale=0.2, n_kv_heads=Hq)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("int8", [False, True])
def test_paged_equals_contiguous(int8):
    rng = np.random.default_rng(12)
    B, Hq, Hkv, D, P = 3, 4, 2, 64, 16
    lens = [37, 16, 70]
    cap = max(lens)
    q, k, v = contiguous_case(rng, B, Hq, Hkv, D, cap)
    kw_c, kw_p = {}, {}
    if int8:
        v, sc = oracle.pack_v_int8(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32))
        kw_c["v_scales"] = sc
    win = [0, 5, 50]
    want = oracle.decode(q, k, v, lens, scale=0.15, n_kv_heads=Hkv, window=win, **kw_c)
    bt = make_table(lens, P, -(-cap // P), rng)
    if int8:
        kw_p["v_scales"] = scatter_pages(sc, lens, P, bt)
    got = oracle.decode(q, scatter_pages(k, lens, P, bt), scatter_pages(v, lens, P, bt), lens,
                        scale=0.15, n_kv_heads=Hkv, window=win, block_table=bt, page_size=P,
                        **kw_p)
    np.testing.assert_array_equal(got, want)


def test_int8_v_matches_dequantised_fp_path():
    """int8 codes * scale enter the sum exactly as the dequantised values would."""
    rng = np.random.default_rng(13)
    B, Hq, Hkv, D, L = 1, 2, 1, 64, 30
    q, k, _ = contiguous_case(rng, B, Hq, Hkv, D, L)
    x = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    codes, sc = oracle.pack_v_int8(x)
    got = oracle.decode(q, k, codes, [L], scale=0.1, n_kv_heads=Hkv, v_scales=sc)
    deq = codes.astype(np.float64) * np.repeat(sc.astype(np.float64), 32, axis=-1)
    for h in range(Hq):
        want = brute_force(q[0, h], k[0, 0], deq[0, 0], 0.1, 0, L)
        np.testing.assert_allclose(got[0, h], want, rtol=1e-12, atol=1e-13)


def test_rows_subset_matches_full():
    rng = np.random.default_rng(14)
    q, k, v = contiguous_case(rng, 3, 4, 2, 32, 20)
    full = oracle.decode(q, k, v, [20, 3, 11], scale=0.5, n_kv_heads=2)
    rows = [11, 0, 5]
    sub = oracle.decode(q, k, v, [20, 3, 11], scale=0.5, n_kv_heads=2, rows=rows)
    for i, r in enumerate(rows):
        np.testing.assert_array_equal(sub[i], full[r // 4, r % 4])


def test_gather_matches_fancy_indexing():
    rng = np.random.default_rng(15)
    B, Hkv, D, P = 3, 2, 16, 16
    lens = [45, 16, 3]
    cache = f16(rng.standard_normal((B, Hkv, max(lens), D)))
    pages, bt = to_paged(cache, lens, P, rng)
    for b in range(B):
        dense = oracle.gather_rows(pages, bt, b, lens[b], n_kv_heads=Hkv, page_size=P)
        t = np.arange(lens[b])
        want = pages[bt[b, t // P], :, t % P].transpose(1, 0, 2)
        np.testing.assert_array_equal(dense.view(np.uint16), want.view(np.uint16))
        np.testing.assert_array_equal(dense, cache[b, :, :lens[b]])


def test_rejects_bad_arguments():
    rng = np.random.default_rng(16)
    q, k, v = contiguous_case(rng, 1, 3, 2, 32, 4)
    with pytest.raises(oracle.OracleError):
        oracle.decode(q, k, v, [4], scale=1.0, n_kv_heads=2)     # 3 % 2 != 0
    q, k, v = contiguous_case(rng, 1, 2, 2, 32, 4)
    with pytest.raises(oracle.OracleError):
        oracle.decode(q, k, v, [5], scale=1.0, n_kv_heads=2)     # L > capacity
