"""GPU parity at the edges of the softmax's numeric range.

- A zero scale makes every attended key weigh the same (the output is the
  mean of the value rows).
- A very large scale spreads the logits over thousands, so almost every
  weight underflows to zero next to the few largest: the kernel must give
  zeros there, not NaN, in the online rescale and in the merge of split
  partials alike.
- A crafted key sits about 90 (natural log units) below the maximum, so its
  weight relative to the maximum is a subnormal fp32 value: the cells near
  FLT_MIN where a product of weight and value could go wrong.

Each case is compared with the fp64 oracle on the same inputs, for both
split kernels.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, to_cuda

pytestmark = pytest.mark.gpu


def W(name, B, Hq, Hkv, D, **kw):
    return Workload(name, B, Hq, Hkv, D, seed=9000 + zlib.crc32(name.encode()) % 1000, **kw)


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


def _gpu(wl, inp, scale):
    dinp = to_cuda(inp)
    cap = dinp["max_blocks"] * (wl.page_size if wl.paged else 1)
    ws = binding.alloc_workspace(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, cap)
    ws.view(torch.uint8).fill_(0xFF)
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), device="cuda")
    binding.fa_decode(dinp["q"], dinp["k_cache"], dinp["v_cache"], dinp.get("v_scales"),
                      dinp["block_table"], dinp["seq_lens"], wl.n_q_heads, wl.n_kv_heads,
                      wl.head_dim, scale, dinp["window"], out, batch=wl.batch,
                      page_size=wl.page_size, max_blocks_per_seq=dinp["max_blocks"],
                      num_blocks=dinp["num_blocks"] if wl.paged else 0, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _oracle(wl, inp, scale):
    return oracle.decode(inp["q"].numpy(), inp["k_cache"].numpy(), inp["v_cache"].numpy(),
                         inp["lens"], scale=scale, n_kv_heads=wl.n_kv_heads,
                         v_scales=None if inp.get("v_scales") is None
                         else inp["v_scales"].numpy(),
                         block_table=None if inp["block_table"] is None
                         else inp["block_table"].numpy(),
                         window=None if inp["window"] is None else inp["window"].numpy(),
                         page_size=wl.page_size, max_blocks=inp["max_blocks"])


@pytest.mark.parametrize("paged,int8", [(False, False), (True, False), (True, True)])
def test_zero_scale_weighs_every_key_alike(kernel, paged, int8):
    wl = W(f"scale0_{paged}_{int8}", 3, 8, 2, 128, paged=paged, v_int8=int8)
    lens = [1, 700, 2500]
    inp = build_case(wl, seq_lens=lens, spare_blocks=2 if paged else 0)
    got = _gpu(wl, inp, 0.0)
    assert_close(got, _oracle(wl, inp, 0.0), int8, "scale 0")
    if not int8:
        # the closed form: the mean of the attended value rows
        v = inp["v_cache"].numpy().astype(np.float64)
        for b, L in enumerate(lens):
            if paged:
                bt = inp["block_table"].numpy()[b]
                rows = np.stack([v[bt[t // 16], :, t % 16] for t in range(L)])   # [L][Hkv][D]
            else:
                rows = np.transpose(v[b, :, :L], (1, 0, 2))
            mean = rows.mean(axis=0)                                         # [Hkv][D]
            for h in range(8):
                np.testing.assert_allclose(got[b, h], mean[h // 4], atol=2e-3)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("scale", [8.0, -8.0])
def test_huge_scale_underflows_to_zero_weights_not_nan(kernel, D, scale):
    """Logit spread in the thousands: nearly all weights are exactly zero in
    fp32, per tile, per split and in the merge; the result is finite and
    matches the oracle."""
    wl = W(f"huge_{D}_{scale}", 4, 8, 2, D, paged=True)
    inp = build_case(wl, seq_lens=[3, 160, 3000, 9000], spare_blocks=2)
    got = _gpu(wl, inp, scale)
    assert_close(got, _oracle(wl, inp, scale), False, f"scale {scale}")


def test_subnormal_relative_weight(kernel):
    """One key 90 natural-log units below the best one: its weight relative
    to the maximum (e^-90, about 8e-40) is subnormal in fp32.  Every other
    key is far lower still.  The output is the best key's value row plus a
    negligible share of the second, and finite."""
    wl = W("subnormal", 1, 4, 1, 128)
    L = 4000
    inp = build_case(wl, seq_lens=[L])
    q = np.zeros((1, 4, 128), dtype=np.float16)
    q[0, :, 0] = 1.0
    k = np.zeros_like(inp["k_cache"].numpy())
    k[0, 0, :L, 0] = -400.0          # every key far below ...
    k[0, 0, 1234, 0] = 100.0         # ... the best one,
    k[0, 0, 2345, 0] = 10.0          # and one 90 below it
    inp["q"] = torch.from_numpy(q)
    inp["k_cache"] = torch.from_numpy(k)
    got = _gpu(wl, inp, 1.0)
    want = _oracle(wl, inp, 1.0)
    assert_close(got, want, False, "subnormal weight")
    v = inp["v_cache"].numpy().astype(np.float64)
    for h in range(4):
        np.testing.assert_allclose(got[0, h], v[0, 0, 1234], atol=1e-6)
