"""The allocation-free entry point (fa_decode_noalloc) against fa_decode.

fa_decode_noalloc serves callers that cannot allocate device memory: it runs
the same kernels with their split-K scratch in a fixed array inside the
library.  This file is collected last so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes
import re

import numpy as np
import pytest
import torch

from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, gpu_decode, oracle_decode, to_cuda

pytestmark = pytest.mark.gpu

# scratch limit compiled into the library (include/fa_decode.h)
NOALLOC_BYTES = 8 << 20


def _noalloc(wl, d):
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    binding.fa_decode_noalloc(d["q"], d["k_cache"], d["v_cache"], d.get("v_scales"),
                              d["block_table"], d["seq_lens"], wl.n_q_heads, wl.n_kv_heads,
                              wl.head_dim, wl.scale, d["window"], out, batch=wl.batch,
                              page_size=wl.page_size, max_blocks_per_seq=d["max_blocks"],
                              num_blocks=d["num_blocks"] if wl.paged else 0)
    return out


@pytest.mark.parametrize("paged", [True, False])
@pytest.mark.parametrize("v_int8", [False, True])
def test_noalloc_matches_fa_decode_on_two_calls_in_a_row(v_int8, paged):
    """Two calls in a row through the C ABI, each compared with fa_decode on
    the same inputs and, independently of both, with the fp64 oracle; paged
    and contiguous caches (the contiguous capacity a multiple of 16)."""
    wl = Workload("noalloc", 4, 16, 4, 128, paged=paged, v_int8=v_int8, window=1000,
                  window_odd_only=True, seed=4242 + 2 * paged + v_int8)
    # the first call uses long sequences (many splits), the second short and
    # ragged ones, so the second reads only scratch it wrote itself
    for lens in ([9000, 12000, 7000, 16000], [300, 17, 5000, 1]):
        inp = build_case(wl, seq_lens=lens, capacity=16000)
        d = to_cuda(inp)
        cap = d["max_blocks"] * (wl.page_size if paged else 1)
        assert binding.fa_decode_workspace_size(4, 16, 4, 128, cap) > 0   # scratch is used
        want = gpu_decode(wl, d).cpu().numpy()
        got = _noalloc(wl, d)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        assert_close(got, want, v_int8, f"noalloc vs fa_decode lens={lens}")
        assert_close(got, oracle_decode(wl, inp), v_int8, f"noalloc vs oracle lens={lens}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    B, Hq, Hkv, D, cap = 256, 64, 8, 256, 1 << 20
    bound = binding.fa_decode_workspace_size(B, Hq, Hkv, D, cap)
    assert bound > NOALLOC_BYTES
    lib = binding.load()
    A = 1 << 20   # never dereferenced: the call must fail before any launch
    rc = lib.fa_decode_noalloc(A, 2 * A, 3 * A, None, None, 4 * A, Hq, Hkv, D, 0.06, None,
                               5 * A, B, 16, cap, 0, None)
    assert rc == -4
    msg = lib.fa_decode_last_error().decode()
    # the message states the call's own need (at most the bound over both V
    # types) and the scratch size
    need = [int(x) for x in re.findall(r"need (\d+) bytes", msg)]
    assert need and NOALLOC_BYTES < need[0] <= bound and str(NOALLOC_BYTES) in msg


def test_noalloc_takes_the_calls_own_need():
    """64 sequences x 4 KV heads (8 query heads each) at a 32K capacity, fp16
    V: the call needs about 6 MB of scratch, while the bound over both V types
    (int8 V at head_dim 128 runs more warps, so more partial slots) is above
    the 8 MiB the library holds.  The call runs, and matches fa_decode."""
    B, Hq, Hkv, D = 64, 32, 4, 128
    wl = Workload("noalloc_big", B, Hq, Hkv, D, paged=True, seed=4343)
    lens = [(i * 37) % 200 + 1 for i in range(B)]
    inp = build_case(wl, seq_lens=lens, capacity=32768)
    d = to_cuda(inp)
    cap = d["max_blocks"] * wl.page_size
    assert binding.fa_decode_workspace_size(B, Hq, Hkv, D, cap) > NOALLOC_BYTES
    want = gpu_decode(wl, d).cpu().numpy()
    got = _noalloc(wl, d)
    torch.cuda.synchronize()
    assert_close(got.cpu().numpy(), want, False, "noalloc at a large capacity")
