"""GPU checks of two properties the decode call promises its callers.

- The workspace needs no initialisation and may be reused, uncleared, across
  calls of other lengths and other shapes.
- A call captured in a CUDA graph (its split kernel and the merge kernel
  launched behind it with programmatic dependent launch, or the one clustered
  launch of a small step) replays correctly with new device-side lengths,
  since the split plan is made on the device.
"""
import zlib

import numpy as np
import pytest
import torch

from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, oracle_decode, to_cuda

pytestmark = pytest.mark.gpu


def W(name, B, Hq, Hkv, D, **kw):
    return Workload(name, B, Hq, Hkv, D, seed=8000 + zlib.crc32(name.encode()) % 1000, **kw)


def _call(wl, dinp, ws, out, stream=None):
    binding.fa_decode(dinp["q"], dinp["k_cache"], dinp["v_cache"], dinp.get("v_scales"),
                      dinp["block_table"], dinp["seq_lens"], wl.n_q_heads, wl.n_kv_heads,
                      wl.head_dim, wl.scale, dinp["window"], out, batch=wl.batch,
                      page_size=wl.page_size, max_blocks_per_seq=dinp["max_blocks"],
                      num_blocks=dinp["num_blocks"] if wl.paged else 0, workspace=ws,
                      stream=stream)


def _with_lens(inp, lens):
    """The same inputs with other lengths (all within the cache as built)."""
    other = dict(inp)
    other["lens"] = list(lens)
    other["seq_lens"] = torch.tensor(lens, dtype=torch.int32)
    return other


def test_workspace_reused_across_calls_and_shapes():
    """One workspace, never cleared, serves calls of different lengths and
    shapes in turn: nothing read in a call comes from an earlier one."""
    a = W("reuse_a", 4, 8, 2, 128, paged=True)
    b = W("reuse_b", 3, 4, 2, 256)
    ia = build_case(a, seq_lens=[3000, 17, 900, 5000], spare_blocks=2)
    ib = build_case(b, seq_lens=[2500, 1, 4000])
    da, db = to_cuda(ia), to_cuda(ib)
    need = max(binding.fa_decode_workspace_size(4, 8, 2, 128, da["max_blocks"] * 16),
               binding.fa_decode_workspace_size(3, 4, 2, 256, db["max_blocks"]))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    # later lengths stay within the first ones: rows past those are NaN
    steps = [(a, ia, da, None), (b, ib, db, None), (a, ia, da, [2999, 16, 0, 4100]),
             (a, ia, da, None), (b, ib, db, [1200, 1, 3]), (b, ib, db, None)]
    for i, (wl, inp, dinp, lens) in enumerate(steps):
        if lens is not None:
            inp = _with_lens(inp, lens)
            dinp = dict(dinp)
            dinp["seq_lens"] = inp["seq_lens"].cuda()
        out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), device="cuda")
        _call(wl, dinp, ws, out)
        assert_close(out.cpu().numpy(), oracle_decode(wl, inp), False, f"call {i} ({wl.name})")


# the stream-K plan (split and merge kernels) and, at small capacities, the
# cluster plan (one clustered launch)
GRAPH_CASES = [(128, False, [4000, 2600, 1500, 3100]), (256, False, [4000, 2600, 1500, 3100]),
               (256, True, [4000, 2600, 1500, 3100]), (128, False, [2000, 1300, 700, 1500]),
               (128, True, [2000, 1300, 700, 1500]), (256, False, [500, 300, 100, 512])]


@pytest.mark.parametrize("D,v_int8,full", GRAPH_CASES)
def test_graph_replay_with_new_lengths(D, v_int8, full):
    """A launch captured in a CUDA graph replays with the lengths the device
    holds at replay time; each replay matches the oracle for those lengths."""
    wl = W(f"graph_{D}_{int(v_int8)}_{max(full)}", 4, 8, 2, D, paged=True, v_int8=v_int8,
           window=700, window_odd_only=True)
    inp = build_case(wl, seq_lens=full, spare_blocks=2)
    dinp = to_cuda(inp)
    cap = dinp["max_blocks"] * wl.page_size
    ws = binding.alloc_workspace(4, 8, 2, D, cap)
    ws.fill_(0xFF)
    out = torch.zeros((4, 8, D), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _call(wl, dinp, ws, out, stream=s)            # first call outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _call(wl, dinp, ws, out, stream=s)
    for lens in (full, [1, full[1] - 1, 0, full[3] - 100], [full[0] - 1, 16, full[2], 17], full):
        dinp["seq_lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert_close(got, oracle_decode(wl, _with_lens(inp, lens)), v_int8, f"replay {lens}")
        for b, L in enumerate(lens):
            if L == 0:
                assert np.all(got[b] == 0)
