"""GPU cache append (fa_append_kv) against the oracle's append, bit for bit,
and append-then-decode against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, gpu_decode, to_cuda

pytestmark = pytest.mark.gpu


def _case(paged, int8, D, seed, extremes=True):
    wl = Workload("append", 4, 8, 2, D, paged=paged, v_int8=int8, seed=seed)
    inp = build_case(wl, seq_lens=[40, 63, 1, 17], capacity=64, spare_blocks=2, poison=False)
    g = torch.Generator().manual_seed(seed + 1)
    kn = torch.randn((4, 2, D), generator=g)
    vn = torch.randn((4, 2, D), generator=g)
    if extremes:   # rounding edge cases, including fp16 overflow to inf
        kn[1, 0, :8] = torch.tensor([65519.0, 65520.0, -1e-8, 3e-5, 1e5, -0.0, 2049.0, 6.1e-5])
    return wl, inp, kn, vn


def _gpu_append(wl, inp, kn, vn, pos):
    d = to_cuda(inp)
    binding.fa_append_kv(kn.cuda(), vn.cuda(), d["k_cache"], d["v_cache"], d.get("v_scales"),
                         d["block_table"], torch.tensor(pos, dtype=torch.int32, device="cuda"),
                         n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim, page_size=wl.page_size,
                         max_blocks_per_seq=inp["max_blocks"],
                         num_blocks=inp["num_blocks"] if wl.paged else 0)
    torch.cuda.synchronize()
    return d


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("D", [128, 256])
def test_append_bit_exact(paged, int8, D):
    wl, inp, kn, vn = _case(paged, int8, D, 100 + D + 2 * paged + int8)
    pos = [40, 63, 1, 17]
    d = _gpu_append(wl, inp, kn, vn, pos)
    k2, v2, s2 = oracle.append_kv(kn.numpy(), vn.numpy(), inp["k_cache"].numpy(),
                                  inp["v_cache"].numpy(), pos,
                                  v_scales=None if not int8 else inp["v_scales"].numpy(),
                                  block_table=None if not paged else inp["block_table"].numpy(),
                                  page_size=wl.page_size, max_blocks=inp["max_blocks"],
                                  num_blocks=inp["num_blocks"] if paged else 0)
    assert d["k_cache"].cpu().numpy().view(np.uint16).tobytes() == k2.view(np.uint16).tobytes()
    assert d["v_cache"].cpu().numpy().tobytes() == v2.tobytes()
    if int8:
        assert d["v_scales"].cpu().numpy().view(np.uint16).tobytes() == \
            s2.view(np.uint16).tobytes()


def test_append_out_of_range_is_skipped_and_flagged():
    wl, inp, kn, vn = _case(True, False, 128, 7)
    inp["block_table"][3, 1] = 10 ** 6                # sequence 3 writes page 1: unmapped
    binding.fa_decode_device_status()
    d = _gpu_append(wl, inp, kn, vn, [-1, 64, 5, 17])
    st = binding.fa_decode_device_status()
    assert st & binding.FA_STATUS_POS_RANGE
    assert st & binding.FA_STATUS_BAD_BLOCK
    k2, v2, _ = oracle.append_kv(kn.numpy(), vn.numpy(), inp["k_cache"].numpy(),
                                 inp["v_cache"].numpy(), [-1, 64, 5, 17],
                                 block_table=inp["block_table"].numpy(), page_size=16,
                                 max_blocks=inp["max_blocks"], num_blocks=inp["num_blocks"])
    assert d["k_cache"].cpu().numpy().view(np.uint16).tobytes() == k2.view(np.uint16).tobytes()
    assert d["v_cache"].cpu().numpy().view(np.uint16).tobytes() == v2.view(np.uint16).tobytes()


@pytest.mark.parametrize("int8", [False, True])
def test_append_then_decode(int8):
    wl, inp, kn, vn = _case(True, int8, 128, 55 + int8, extremes=False)
    pos = [40, 63, 1, 17]
    d = _gpu_append(wl, inp, kn, vn, pos)
    k2, v2, s2 = oracle.append_kv(kn.numpy(), vn.numpy(), inp["k_cache"].numpy(),
                                  inp["v_cache"].numpy(), pos,
                                  v_scales=None if not int8 else inp["v_scales"].numpy(),
                                  block_table=inp["block_table"].numpy(), page_size=16,
                                  max_blocks=inp["max_blocks"], num_blocks=inp["num_blocks"])
    lens = [t + 1 for t in pos]
    d["seq_lens"] = torch.tensor(lens, dtype=torch.int32, device="cuda")
    got = gpu_decode(wl, d).cpu().numpy()
    want = oracle.decode(inp["q"].numpy(), k2, v2, lens, scale=wl.scale, n_kv_heads=2,
                         v_scales=s2, block_table=inp["block_table"].numpy(), page_size=16)
    assert_close(got, want, int8, "append then decode")
