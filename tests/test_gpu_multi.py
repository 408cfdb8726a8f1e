"""Multi-query decode (fa_decode_multi) against the oracle's multi-query mode.
Columns of the tensor-core tile are (query, head) pairs, so the cases cover
one and several column groups, windows that leave a column with no key in a
whole tile, int8 V, and sequences shorter than the number of queries."""
import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, to_cuda

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, Hq, Hkv, D, Tq, window, paged, int8, lens
    ("g4_tq2", 3, 8, 2, 128, 2, 0, True, False, [100, 1000, 17]),
    ("g4_tq4_window", 3, 8, 2, 128, 4, 5, True, False, [100, 1000, 40]),
    ("g4_tq7_window40", 2, 8, 2, 128, 7, 40, False, False, [300, 64]),
    ("g8_tq3_groups", 2, 16, 2, 128, 3, 0, True, False, [500, 33]),
    ("g2_d256_tq3", 3, 4, 2, 256, 3, 0, True, False, [200, 2000, 9]),
    ("g2_d256_tq5_int8", 2, 4, 2, 256, 5, 64, True, True, [700, 100]),
    ("g4_tq4_int8_contig", 2, 8, 2, 128, 4, 0, False, True, [96, 48]),
    ("short_seqs", 3, 8, 2, 128, 6, 0, True, False, [2, 6, 1]),
    ("g1_tq8", 2, 2, 2, 128, 8, 0, True, False, [64, 1000]),
    ("g2_d256_tq8", 3, 4, 2, 256, 8, 0, True, False, [900, 2000, 5]),
    ("g2_d256_tq6_window_contig", 2, 4, 2, 256, 6, 50, False, False, [300, 64]),
    ("g4_d256_tq7_ragged", 5, 8, 2, 256, 7, 0, True, False, [1, 7, 33, 1500, 4000]),
    # 40 x 4 x 8 = 1280 output rows: at or above four rows per SM the merge
    # takes a warp per row
    ("many_rows_tq4", 40, 8, 2, 128, 4, 30, True, False,
     [(i * 97) % 700 + (i % 3) for i in range(40)]),
    ("many_rows_d256_tq3_int8", 26, 8, 2, 256, 3, 0, True, True,
     [(i * 131) % 900 + 1 for i in range(26)]),
]

# The same kind of cases with a block table of 2^20 tokens per sequence: the
# K/V the capacity allows passes the two-column-group threshold, so units
# hold 16 columns (at D=256 with the query rows in shared memory, fp16 or int8
# V), while the pool holds only the blocks the lengths need.
BIG_CAP = 1 << 20
CASES_TWO_GROUPS = [
    ("2g_g4_tq4_window", 3, 8, 2, 128, 4, 5, True, False, [100, 1000, 40]),
    ("2g_g8_tq3", 2, 16, 2, 128, 3, 0, True, False, [500, 33]),
    ("2g_g4_tq4_int8", 3, 8, 2, 128, 4, 0, True, True, [96, 1500, 7]),
    ("2g_d256_tq8", 3, 4, 2, 256, 8, 0, True, False, [900, 2000, 5]),
    ("2g_d256_tq6_window", 2, 4, 2, 256, 6, 50, True, False, [300, 64]),
    ("2g_d256_tq7_ragged", 5, 8, 2, 256, 7, 0, True, False, [1, 7, 33, 1500, 4000]),
    ("2g_d256_tq8_int8", 3, 4, 2, 256, 8, 0, True, True, [900, 2000, 5]),
    ("2g_d256_tq5_int8_window", 4, 8, 2, 256, 5, 40, True, True, [1, 300, 2500, 64]),
]


ALL_CASES = [c + (None,) for c in CASES] + [c + (BIG_CAP,) for c in CASES_TWO_GROUPS]


@pytest.mark.parametrize("case", ALL_CASES, ids=[c[0] for c in ALL_CASES])
def test_multi_query_matches_oracle(case):
    name, B, Hq, Hkv, D, Tq, window, paged, int8, lens, big_cap = case
    wl = Workload(name, B, Hq, Hkv, D, paged=paged, v_int8=int8, window=window,
                  seed=900 + len(name))
    cap = big_cap or max(lens)
    if not paged:
        cap = -(-cap // 16) * 16
    inp = build_case(wl, seq_lens=lens, capacity=cap, spare_blocks=2 if paged else 0)
    g = np.random.default_rng(len(name))
    q = g.standard_normal((B, Tq, Hq, D)).astype(np.float16)
    want = oracle.decode_multi(q, inp["k_cache"].numpy(), inp["v_cache"].numpy(), lens,
                               scale=wl.scale, n_kv_heads=Hkv,
                               v_scales=None if not int8 else inp["v_scales"].numpy(),
                               block_table=None if not paged else inp["block_table"].numpy(),
                               window=None if inp["window"] is None else inp["window"].numpy(),
                               page_size=16, max_blocks=inp["max_blocks"])
    d = to_cuda(inp)
    n = binding.fa_decode_multi_workspace_size(B, Tq, Hq, Hkv, D,
                                               inp["max_blocks"] * (16 if paged else 1))
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, Tq, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_multi(torch.from_numpy(q).cuda(), d["k_cache"], d["v_cache"],
                            d.get("v_scales"), d["block_table"], d["seq_lens"], Hq, Hkv, D,
                            wl.scale, d["window"], out, max_blocks_per_seq=inp["max_blocks"],
                            num_blocks=inp["num_blocks"] if paged else 0, workspace=ws)
    got = out.cpu().numpy()
    assert_close(got, want, int8, name)
    for b, L in enumerate(lens):
        for j in range(Tq):
            if L - Tq + j < 0:
                assert np.all(got[b, j] == 0)


def test_single_query_through_multi_equals_fa_decode():
    wl = Workload("tq1", 3, 8, 2, 128, paged=True, window=100, seed=31)
    inp = build_case(wl, seq_lens=[700, 50, 3000])
    d = to_cuda(inp)
    cap = inp["max_blocks"] * 16
    ws = binding.alloc_workspace(3, 8, 2, 128, cap)
    a = torch.empty((3, 8, 128), device="cuda")
    binding.fa_decode(d["q"], d["k_cache"], d["v_cache"], None, d["block_table"], d["seq_lens"],
                      8, 2, 128, wl.scale, d["window"], a, workspace=ws)
    n = binding.fa_decode_multi_workspace_size(3, 1, 8, 2, 128, cap)
    ws2 = torch.empty((max(n, 16),), dtype=torch.uint8, device="cuda")
    b = torch.empty((3, 1, 8, 128), device="cuda")
    binding.fa_decode_multi(d["q"].unsqueeze(1).contiguous(), d["k_cache"], d["v_cache"], None,
                            d["block_table"], d["seq_lens"], 8, 2, 128, wl.scale, d["window"], b,
                            workspace=ws2)
    assert torch.equal(a, b[:, 0])
