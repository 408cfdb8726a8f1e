"""Ring-cache decode (fa_decode_ring) and append (fa_append_kv_ring) against
the oracle's ring mode.  Rows a ring has never written are NaN."""
import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding

from _helpers import assert_close

pytestmark = pytest.mark.gpu


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


def _ring_case(seed, B, Hq, Hkv, D, C, n_seen, int8):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, C, D)).astype(np.float16)
    if int8:
        v, sc = oracle.pack_v_int8(rng.standard_normal((B, Hkv, C, D)).astype(np.float32))
    else:
        v, sc = rng.standard_normal((B, Hkv, C, D)).astype(np.float16), None
    for b, n in enumerate(n_seen):          # rows never written yet
        if n < C:
            k[b, :, n:] = np.nan
            if not int8:
                v[b, :, n:] = np.nan
            else:
                sc[b, :, n:] = np.nan
    return q, k, v, sc


@pytest.mark.parametrize("D,C", [(128, 64), (256, 32), (128, 256)])
@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("window", [0, 10, 40])
def test_ring_decode_matches_oracle(D, C, int8, window, kernel):
    B, Hq, Hkv = 5, 8, 2
    n_seen = [7, C, C + 5, 3 * C + 9, C + 16]
    q, k, v, sc = _ring_case(1000 + D + C + window + int8, B, Hq, Hkv, D, C, n_seen, int8)
    win = [window] * B
    want = oracle.decode_ring(q, k, v, n_seen, scale=D ** -0.5, n_kv_heads=Hkv, v_scales=sc,
                              window=win)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = binding.fa_decode_workspace_size(B, Hq, Hkv, D, C + 16)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_ring(t(q), t(k), t(v), t(sc), t(np.array(n_seen, dtype=np.int32)), Hq, Hkv,
                           D, D ** -0.5, t(np.array(win, dtype=np.int32)), out, workspace=ws)
    assert_close(out.cpu().numpy(), want, int8, f"ring D={D} C={C} w={window}")


@pytest.mark.parametrize("int8", [False, True])
def test_ring_append_bit_exact_then_decode(int8):
    B, Hq, Hkv, D, C = 4, 8, 2, 128, 64
    n_seen = [10, 63, 64, 200]              # the new token's position is n_seen[b]
    q, k, v, sc = _ring_case(77 + int8, B, Hq, Hkv, D, C, n_seen, int8)
    g = np.random.default_rng(5)
    kn = g.standard_normal((B, Hkv, D)).astype(np.float32)
    vn = g.standard_normal((B, Hkv, D)).astype(np.float32)
    k2, v2, s2 = oracle.append_kv_ring(kn, vn, k, v, n_seen, v_scales=sc)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    dk, dv, ds = t(k), t(v), t(sc)
    binding.fa_append_kv_ring(t(kn), t(vn), dk, dv, ds, t(np.array(n_seen, dtype=np.int32)))
    torch.cuda.synchronize()
    assert dk.cpu().numpy().view(np.uint16).tobytes() == k2.view(np.uint16).tobytes()
    assert dv.cpu().numpy().tobytes() == v2.tobytes()
    if int8:
        assert ds.cpu().numpy().view(np.uint16).tobytes() == s2.view(np.uint16).tobytes()
    lens = [n + 1 for n in n_seen]
    want = oracle.decode_ring(q, k2, v2, lens, scale=0.1, n_kv_heads=Hkv, v_scales=s2)
    n = binding.fa_decode_workspace_size(B, Hq, Hkv, D, C + 16)
    ws = torch.empty((max(n, 16),), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, D), device="cuda")
    binding.fa_decode_ring(t(q), dk, dv, ds, t(np.array(lens, dtype=np.int32)), Hq, Hkv, D, 0.1,
                           None, out, workspace=ws)
    assert_close(out.cpu().numpy(), want, int8, "ring append then decode")
