"""The cluster plan of small steps: one thread-block cluster per (sequence,
KV head) unit, the unit's tiles split over the cluster's warps, the warps'
partials folded through distributed shared memory, and no merge kernel.

Every case is compared with the oracle twice: under the plan the library
picks and with the plan held to stream-K (FA_DECODE_PLAN=streamk).  The
workspace is filled with 0xFF (NaN floats) before each call; the cluster plan
writes nothing there, so an untouched workspace shows that plan ran."""
import numpy as np
import pytest
import torch

from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, oracle_decode, to_cuda

pytestmark = pytest.mark.gpu

W = Workload
CASES = [
    # the 1 x 512 decode shape: two units of 32 tiles, one tile per warp
    (W("one_seq_512", 1, 8, 2, 128, seed=31), [512]),
    # ragged, paged, windowed: units of 1 to 128 tiles, many warps without tiles
    (W("ragged_paged_win", 3, 16, 4, 128, paged=True, window=100, seed=32), [1, 17, 2048]),
    # an empty sequence (its units' outputs are zero rows) and int8 V
    (W("empty_int8", 2, 8, 2, 128, v_int8=True, paged=True, seed=33), [0, 640]),
    # head_dim 256 (at most 512 tokens there), fp16 and int8 V (int8: 8 warps
    # per CTA, 64 partials per unit)
    (W("d256", 2, 8, 4, 256, seed=34), [300, 500]),
    (W("d256_int8", 1, 16, 8, 256, v_int8=True, paged=True, seed=35), [497]),
    # one query head per KV head, and eight
    (W("mha", 2, 4, 4, 128, seed=36), [33, 250]),
    (W("gqa8", 2, 16, 2, 128, paged=True, window=64, seed=37), [1024, 65]),
    # more units than 8-CTA clusters fit: 4-CTA clusters (64 units), then 2-CTA
    # clusters (128 units), each warp still at most 4 tiles
    (W("clusters_of_4", 8, 32, 8, 128, paged=True, seed=39), [1000, 3, 512, 1024, 0, 77, 640, 999]),
    (W("clusters_of_2", 16, 32, 8, 128, seed=40), [512, 1, 300, 17, 480, 512, 0, 256,
                                                   100, 511, 64, 33, 200, 400, 16, 500]),
    # 256 units of at most 16 tiles: one-CTA clusters, the columns folded in two passes
    (W("clusters_of_1", 32, 32, 8, 128, paged=True, window=100, window_odd_only=True, seed=41),
     [256, 1, 0, 17, 255, 128, 64, 200] * 4),
    # int8 V at head_dim 128 runs 3 CTAs per SM, so more clusters fit at each size than with
    # fp16 V: the same kinds of steps with int8 V, paged and contiguous
    (W("int8_many_units", 16, 32, 8, 128, v_int8=True, paged=True, seed=42),
     [512, 1, 300, 17, 480, 512, 0, 256, 100, 511, 64, 33, 200, 400, 16, 500]),
    (W("int8_small_units", 32, 32, 8, 128, v_int8=True, window=50, seed=43),
     [256, 1, 0, 17, 255, 128, 64, 200] * 4),
]


def _call(wl, d, ws):
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), device="cuda")
    binding.fa_decode(d["q"], d["k_cache"], d["v_cache"], d.get("v_scales"), d["block_table"],
                      d["seq_lens"], wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.scale,
                      d["window"], out, batch=wl.batch, page_size=wl.page_size,
                      max_blocks_per_seq=d["max_blocks"],
                      num_blocks=d["num_blocks"] if wl.paged else 0, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("wl,lens", CASES, ids=[w.name for w, _ in CASES])
def test_cluster_plan_matches_oracle_and_writes_no_partials(wl, lens, monkeypatch):
    monkeypatch.setenv("FA_DECODE_KERNEL", "mma")
    cap = -(-max(max(lens), 1) // 16) * 16
    inp = build_case(wl, seq_lens=lens, capacity=cap, spare_blocks=2 if wl.paged else 0)
    d = to_cuda(inp)
    want = oracle_decode(wl, inp)
    n = binding.fa_decode_workspace_size(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                                         d["max_blocks"] * (wl.page_size if wl.paged else 1))
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")

    monkeypatch.delenv("FA_DECODE_PLAN", raising=False)
    got = _call(wl, d, ws)
    assert_close(got, want, wl.v_int8, f"{wl.name} cluster plan")
    assert bool((ws == 0xFF).all()), "the cluster plan wrote to the workspace"
    # the same call again: the same bytes (the fold order is fixed)
    assert np.array_equal(_call(wl, d, ws), got)

    monkeypatch.setenv("FA_DECODE_PLAN", "streamk")
    got_sk = _call(wl, d, ws)
    assert_close(got_sk, want, wl.v_int8, f"{wl.name} stream-K plan")
    if wl.name == "one_seq_512":
        # stream-K splits each 32-tile unit over many warps: partials in the workspace
        assert not bool((ws == 0xFF).all())


def test_cluster_plan_flags_bad_blocks_and_clamped_lengths(monkeypatch):
    monkeypatch.setenv("FA_DECODE_KERNEL", "mma")
    monkeypatch.delenv("FA_DECODE_PLAN", raising=False)
    wl = W("flags", 2, 8, 2, 128, paged=True, seed=38)
    inp = build_case(wl, seq_lens=[200, 90], capacity=208, spare_blocks=1, poison=False)
    want = oracle_decode(wl, inp)                       # before the table is broken below
    inp["block_table"][1, 2] = 10 ** 6                  # sequence 1's third page: unmapped
    d = to_cuda(inp)
    d["seq_lens"] = torch.tensor([200, 5000], dtype=torch.int32, device="cuda")  # beyond capacity
    n = binding.fa_decode_workspace_size(2, 8, 2, 128, d["max_blocks"] * 16)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    binding.fa_decode_device_status()
    out = _call(wl, d, ws)
    st = binding.fa_decode_device_status()
    assert st & binding.FA_STATUS_BAD_BLOCK
    assert st & binding.FA_STATUS_LEN_CLAMPED
    assert np.all(np.isfinite(out[0]))
    assert_close(out[:1], want[:1], False, "flags: the healthy sequence")
