"""Slot-map decode (fa_decode_slots) and append (fa_append_kv_slots) against
the oracle's slot map: the active rows name a permuted subset of a larger
pool of per-slot caches.  Every cache row the step must not read (idle slots,
rows past a slot's length) holds NaN, so reading the wrong slot fails."""
import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding

from _helpers import assert_close

pytestmark = pytest.mark.gpu

N_SLOTS = 64


@pytest.fixture(params=["mma", "mma_streamk", "simt"])
def kernel(request, monkeypatch):
    """Run a case through each split kernel and plan: the tensor-core kernel
    with the plan the library picks (the cluster plan for small steps), the
    tensor-core kernel held to the stream-K plan (FA_DECODE_PLAN=streamk), and
    the CUDA-core kernel (FA_DECODE_KERNEL=simt); int8 V cases included."""
    monkeypatch.setenv("FA_DECODE_KERNEL", "simt" if request.param == "simt" else "mma")
    if request.param == "mma_streamk":
        monkeypatch.setenv("FA_DECODE_PLAN", "streamk")
    else:
        monkeypatch.delenv("FA_DECODE_PLAN", raising=False)
    return request.param


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _pool(seed, Hkv, C, D, int8, lens_by_slot, ring):
    """A pool [N_SLOTS, Hkv, C, D]; rows a slot has not written are NaN."""
    rng = np.random.default_rng(seed)
    k = np.full((N_SLOTS, Hkv, C, D), np.nan, dtype=np.float16)
    if int8:
        v, sc = oracle.pack_v_int8(rng.standard_normal((N_SLOTS, Hkv, C, D)).astype(np.float32))
        sc = sc.copy()
        sc[:] = np.nan
    else:
        v, sc = np.full((N_SLOTS, Hkv, C, D), np.nan, dtype=np.float16), None
    for s, L in lens_by_slot.items():
        n = min(L, C) if ring else L
        k[s, :, :n] = rng.standard_normal((Hkv, n, D)).astype(np.float16)
        if int8:
            codes, scales = oracle.pack_v_int8(rng.standard_normal((Hkv, n, D)).astype(np.float32))
            v[s, :, :n], sc[s, :, :n] = codes, scales
        else:
            v[s, :, :n] = rng.standard_normal((Hkv, n, D)).astype(np.float16)
    return k, v, sc


def _run(q, k, v, sc, slots, lens, win, Hq, Hkv, D, C, ring, scale):
    B = len(slots)
    n = binding.fa_decode_workspace_size(B, Hq, Hkv, D, C + 16 if ring else C)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_slots(_t(q), _t(k), _t(v), _t(sc), _t(np.array(slots, dtype=np.int32)),
                            _t(np.array(lens, dtype=np.int32)), Hq, Hkv, D, scale,
                            None if win is None else _t(np.array(win, dtype=np.int32)), out,
                            ring=ring, workspace=ws)
    return out.cpu().numpy()


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("window", [0, 37])
def test_slots_decode_matches_oracle(D, int8, window, kernel):
    Hq, Hkv, C = 8, 2, 160
    slots = [41, 3, 63, 17, 0, 29, 52, 8]                  # 8 active of 64, permuted
    lens = [160, 1, 75, 0, 144, 16, 99, 33]
    k, v, sc = _pool(300 + D + int8 + window, Hkv, C, D, int8, dict(zip(slots, lens)), False)
    rng = np.random.default_rng(7 + D)
    q = rng.standard_normal((len(slots), Hq, D)).astype(np.float16)
    win = [window] * len(slots)
    want = oracle.decode_slots(q, k, v, lens, slots, scale=D ** -0.5, n_kv_heads=Hkv,
                               v_scales=sc, window=win)
    got = _run(q, k, v, sc, slots, lens, win, Hq, Hkv, D, C, False, D ** -0.5)
    assert_close(got, want, int8, f"slots D={D} int8={int8} w={window}")


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("int8", [False, True])
def test_ring_slots_decode_matches_oracle(D, int8, kernel):
    Hq, Hkv, C = 16, 4, 64
    slots = [60, 2, 31, 47, 9]
    seen = [7, 64, 65, 300, 130]                           # below, at and past capacity
    k, v, sc = _pool(400 + D + int8, Hkv, C, D, int8, dict(zip(slots, seen)), True)
    rng = np.random.default_rng(11 + D)
    q = rng.standard_normal((len(slots), Hq, D)).astype(np.float16)
    win = [0, 0, 20, 50, 0]
    want = oracle.decode_slots(q, k, v, seen, slots, scale=D ** -0.5, n_kv_heads=Hkv,
                               v_scales=sc, window=win, ring=True)
    got = _run(q, k, v, sc, slots, seen, win, Hq, Hkv, D, C, True, D ** -0.5)
    assert_close(got, want, int8, f"ring slots D={D} int8={int8}")


def test_slot_out_of_range_gives_zero_row_and_flag():
    Hq, Hkv, D, C = 8, 2, 128, 64
    slots = [5, 64, -1, 12]
    lens = [64, 64, 64, 30]
    k, v, sc = _pool(500, Hkv, C, D, False, {5: 64, 12: 30}, False)
    q = np.random.default_rng(3).standard_normal((4, Hq, D)).astype(np.float16)
    binding.fa_decode_device_status()
    got = _run(q, k, v, sc, slots, lens, None, Hq, Hkv, D, C, False, 0.1)
    st = binding.fa_decode_device_status()
    assert st & binding.FA_STATUS_BAD_SLOT
    assert np.all(got[1:3] == 0.0)
    want = oracle.decode_slots(q, k, v, lens, slots, scale=0.1, n_kv_heads=Hkv)
    assert_close(got, want, False, "bad slot ids")


@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("int8", [False, True])
def test_append_slots_bit_exact_then_decode(ring, int8):
    Hq, Hkv, D, C = 8, 2, 128, 64
    slots = [33, 6, 50, 21]
    seen = [10, 63, 0, 200] if ring else [10, 63, 0, 40]   # the new token's position
    k, v, sc = _pool(600 + 2 * ring + int8, Hkv, C, D, int8, dict(zip(slots, seen)), ring)
    g = np.random.default_rng(8)
    kn = g.standard_normal((4, Hkv, D)).astype(np.float32)
    vn = g.standard_normal((4, Hkv, D)).astype(np.float32)
    k2, v2, s2 = oracle.append_kv_slots(kn, vn, k, v, slots, seen, v_scales=sc, ring=ring)
    dk, dv, ds = _t(k), _t(v), _t(sc)
    binding.fa_append_kv_slots(_t(kn), _t(vn), dk, dv, ds, _t(np.array(slots, dtype=np.int32)),
                               _t(np.array(seen, dtype=np.int32)), ring=ring)
    torch.cuda.synchronize()
    assert dk.cpu().numpy().view(np.uint16).tobytes() == k2.view(np.uint16).tobytes()
    assert dv.cpu().numpy().tobytes() == v2.tobytes()
    if int8:
        assert ds.cpu().numpy().view(np.uint16).tobytes() == s2.view(np.uint16).tobytes()
    lens = [n + 1 for n in seen]
    q = g.standard_normal((4, Hq, D)).astype(np.float16)
    want = oracle.decode_slots(q, k2, v2, lens, slots, scale=0.1, n_kv_heads=Hkv, v_scales=s2,
                               ring=ring)
    got = _run(q, k2, v2, s2, slots, lens, None, Hq, Hkv, D, C, ring, 0.1)
    assert_close(got, want, int8, f"append slots ring={ring} then decode")


def test_append_slots_out_of_range_is_skipped_and_flagged():
    Hkv, D, C = 2, 128, 32
    k, v, _ = _pool(700, Hkv, C, D, False, {1: 10, 2: 10}, False)
    g = np.random.default_rng(9)
    kn = g.standard_normal((3, Hkv, D)).astype(np.float32)
    vn = g.standard_normal((3, Hkv, D)).astype(np.float32)
    binding.fa_decode_device_status()
    dk, dv = _t(k), _t(v)
    binding.fa_append_kv_slots(_t(kn), _t(vn), dk, dv, None,
                               _t(np.array([1, 64, -3], dtype=np.int32)),
                               _t(np.array([10, 5, 5], dtype=np.int32)))
    st = binding.fa_decode_device_status()
    assert st & binding.FA_STATUS_BAD_SLOT
    k2, v2, _ = oracle.append_kv_slots(kn, vn, k, v, [1, 64, -3], [10, 5, 5])
    assert dk.cpu().numpy().view(np.uint16).tobytes() == k2.view(np.uint16).tobytes()
    assert dv.cpu().numpy().view(np.uint16).tobytes() == v2.view(np.uint16).tobytes()
