"""GPU checks of fa_decode_batch_invariant.

Each sequence's KV range is cut into splits of a fixed number of keys, so a
sequence's output must be the same bytes however it is batched: alone, in
another order, or beside other sequences (the pages' batched-vs-serial
parity rule).  The outputs also match the fp64 oracle within the usual
tolerances.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, oracle_decode, to_cuda

pytestmark = pytest.mark.gpu


def W(name, B, Hq, Hkv, D, **kw):
    return Workload(name, B, Hq, Hkv, D, seed=9500 + zlib.crc32(name.encode()) % 1000, **kw)


def _run(wl, dinp, split_tokens, rows=None):
    """Decode sequences `rows` (default: all) of the case as one batch."""
    rows = list(range(wl.batch)) if rows is None else list(rows)
    idx = torch.tensor(rows, device="cuda")
    q = dinp["q"].index_select(0, idx).contiguous()
    sl = dinp["seq_lens"].index_select(0, idx).contiguous()
    bt = None if dinp["block_table"] is None else dinp["block_table"].index_select(0, idx).contiguous()
    win = None if dinp["window"] is None else dinp["window"].index_select(0, idx).contiguous()
    k, v, vs = dinp["k_cache"], dinp["v_cache"], dinp.get("v_scales")
    if not wl.paged:        # contiguous caches are indexed by position in the batch
        k = k.index_select(0, idx).contiguous()
        v = v.index_select(0, idx).contiguous()
        vs = None if vs is None else vs.index_select(0, idx).contiguous()
    B = len(rows)
    cap = dinp["max_blocks"] * (wl.page_size if wl.paged else 1)
    n = binding.fa_decode_batch_invariant_workspace_size(B, wl.n_q_heads, wl.n_kv_heads,
                                                         wl.head_dim, cap, split_tokens)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, wl.n_q_heads, wl.head_dim), float("nan"), device="cuda")
    binding.fa_decode_batch_invariant(q, k, v, vs, bt, sl, wl.n_q_heads, wl.n_kv_heads,
                                      wl.head_dim, wl.scale, win, out, split_tokens=split_tokens,
                                      batch=B, page_size=wl.page_size,
                                      max_blocks_per_seq=dinp["max_blocks"],
                                      num_blocks=dinp["num_blocks"] if wl.paged else 0,
                                      workspace=ws)
    torch.cuda.synchronize()
    return out.cpu()


CASES = [
    (W("bi_d128_paged", 6, 8, 2, 128, paged=True), [1, 15, 700, 3000, 0, 9000], 512),
    (W("bi_d128_contig_win", 5, 16, 2, 128, window=300, window_odd_only=True),
     [17, 2000, 2000, 513, 4096], 256),
    (W("bi_d256_paged", 4, 8, 4, 256, paged=True), [33, 1024, 5000, 7], 64),
    (W("bi_d256_int8", 4, 8, 2, 256, paged=True, v_int8=True), [2500, 9, 1200, 4000], 512),
    (W("bi_d128_int8_g8", 3, 32, 4, 128, paged=True, v_int8=True, window=1000),
     [6000, 999, 1001], 128),
    (W("bi_d128_split16", 3, 4, 4, 128, paged=True), [100, 257, 40], 16),
]


@pytest.mark.parametrize("wl,lens,st", CASES, ids=[c[0].name for c in CASES])
def test_matches_oracle(wl, lens, st):
    inp = build_case(wl, seq_lens=lens, spare_blocks=2 if wl.paged else 0)
    got = _run(wl, to_cuda(inp), st).numpy()
    assert_close(got, oracle_decode(wl, inp), wl.v_int8, wl.name)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0)


@pytest.mark.parametrize("wl,lens,st", CASES, ids=[c[0].name for c in CASES])
def test_each_sequence_alone_in_another_order_and_in_a_bigger_batch_bitwise(wl, lens, st):
    inp = build_case(wl, seq_lens=lens, spare_blocks=2 if wl.paged else 0)
    dinp = to_cuda(inp)
    whole = _run(wl, dinp, st)
    for b in range(wl.batch):
        alone = _run(wl, dinp, st, rows=[b])
        assert torch.equal(alone[0], whole[b]), f"sequence {b} alone"
    perm = list(reversed(range(wl.batch)))
    shuffled = _run(wl, dinp, st, rows=perm)
    for i, b in enumerate(perm):
        assert torch.equal(shuffled[i], whole[b]), f"sequence {b} reordered"
    twice = _run(wl, dinp, st, rows=list(range(wl.batch)) * 2)
    assert torch.equal(twice[:wl.batch], whole) and torch.equal(twice[wl.batch:], whole)


def test_stream_k_plan_is_batch_dependent_but_close():
    """For contrast: fa_decode's plan cuts a sequence where the batch puts the
    worker boundaries, so its bytes may change with the batch; the results
    still agree within the tolerances."""
    wl, lens, st = CASES[0]
    inp = build_case(wl, seq_lens=lens, spare_blocks=2)
    dinp = to_cuda(inp)
    inv = _run(wl, dinp, st).numpy()
    cap = dinp["max_blocks"] * wl.page_size
    ws = binding.alloc_workspace(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, cap)
    out = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), device="cuda")
    binding.fa_decode(dinp["q"], dinp["k_cache"], dinp["v_cache"], None, dinp["block_table"],
                      dinp["seq_lens"], wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.scale, None,
                      out, workspace=ws)
    assert_close(out.cpu().numpy(), inv, False, "stream-K vs batch-invariant")


def _multi(wl, d, q, tq, st, rows):
    idx = torch.tensor(rows, device="cuda")
    qq = q.index_select(0, idx).contiguous()
    sl = d["seq_lens"].index_select(0, idx).contiguous()
    bt = d["block_table"].index_select(0, idx).contiguous()
    win = None if d["window"] is None else d["window"].index_select(0, idx).contiguous()
    B = len(rows)
    cap = d["max_blocks"] * wl.page_size
    n = binding.fa_decode_multi_batch_invariant_workspace_size(B, tq, wl.n_q_heads, wl.n_kv_heads,
                                                               wl.head_dim, cap, st)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, tq, wl.n_q_heads, wl.head_dim), float("nan"), device="cuda")
    binding.fa_decode_multi_batch_invariant(qq, d["k_cache"], d["v_cache"], d.get("v_scales"), bt,
                                            sl, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                                            wl.scale, win, out, split_tokens=st,
                                            max_blocks_per_seq=d["max_blocks"],
                                            num_blocks=d["num_blocks"], workspace=ws)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("D,int8,tq,st", [(128, False, 3, 256), (256, True, 5, 64)])
def test_multi_query_batch_invariant(D, int8, tq, st):
    """Several queries per sequence (columns beyond 8 span two units): the
    oracle's multi-query mode, and bit-identical rows alone and reordered."""
    wl = W(f"bi_multi_{D}_{int(int8)}", 5, 8, 2, D, paged=True, v_int8=int8, window=400,
           window_odd_only=True)
    lens = [1, 700, 2100, 33, 1300]
    inp = build_case(wl, seq_lens=lens, spare_blocks=2)
    q = np.random.default_rng(D + tq).standard_normal((5, tq, 8, D)).astype(np.float16)
    d = to_cuda(inp)
    qd = torch.from_numpy(q).cuda()
    whole = _multi(wl, d, qd, tq, st, list(range(5)))
    want = oracle.decode_multi(q, inp["k_cache"].numpy(), inp["v_cache"].numpy(), lens,
                               scale=wl.scale, n_kv_heads=2,
                               v_scales=None if not int8 else inp["v_scales"].numpy(),
                               block_table=inp["block_table"].numpy(),
                               window=inp["window"].numpy(), page_size=16,
                               max_blocks=inp["max_blocks"])
    assert_close(whole.numpy(), want, int8, wl.name)
    for b in range(5):
        assert torch.equal(_multi(wl, d, qd, tq, st, [b])[0], whole[b]), f"sequence {b} alone"
    perm = [3, 0, 4, 2, 1]
    got = _multi(wl, d, qd, tq, st, perm)
    for i, b in enumerate(perm):
        assert torch.equal(got[i], whole[b]), f"sequence {b} reordered"


def test_ring_batch_invariant():
    C = 128
    B, Hq, Hkv, D = 4, 8, 2, 128
    seen = [5, 128, 300, 1000]
    g = np.random.default_rng(77)
    q = g.standard_normal((B, Hq, D)).astype(np.float16)
    k = g.standard_normal((B, Hkv, C, D)).astype(np.float16)
    v = g.standard_normal((B, Hkv, C, D)).astype(np.float16)
    win = np.array([0, 50, 0, 100], dtype=np.int32)
    scale = D ** -0.5
    want = oracle.decode_ring(q, k, v, seen, scale=scale, n_kv_heads=Hkv, window=win)
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    sl = torch.tensor(seen, dtype=torch.int32, device="cuda")
    wd = torch.from_numpy(win).cuda()

    def run(rows, st=32):
        idx = torch.tensor(rows, device="cuda")
        n = binding.fa_decode_batch_invariant_workspace_size(len(rows), Hq, Hkv, D, C + 16, st)
        ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
        out = torch.full((len(rows), Hq, D), float("nan"), device="cuda")
        binding.fa_decode_ring_batch_invariant(
            qd.index_select(0, idx).contiguous(), kd.index_select(0, idx).contiguous(),
            vd.index_select(0, idx).contiguous(), None, sl.index_select(0, idx).contiguous(),
            Hq, Hkv, D, scale, wd.index_select(0, idx).contiguous(), out, split_tokens=st,
            workspace=ws)
        torch.cuda.synchronize()
        return out.cpu()

    whole = run(list(range(B)))
    assert_close(whole.numpy(), want, False, "ring batch-invariant")
    for b in range(B):
        assert torch.equal(run([b])[0], whole[b]), f"ring sequence {b} alone"


def test_batch_invariant_flags_clamped_lengths_and_bad_blocks():
    """The batch-invariant plan reads lengths and block ids through the same
    checks: a length beyond capacity is clamped and flagged, a block id out
    of range skips its tile and is flagged, other sequences are unaffected."""
    wl = W("bi_status", 3, 8, 2, 128, paged=True)
    inp = build_case(wl, seq_lens=[64, 32, 500])
    want = oracle_decode(wl, inp)
    dinp = to_cuda(inp)
    binding.fa_decode_device_status()                       # clear
    dinp["seq_lens"] = torch.tensor([64, 10 ** 6, 500], dtype=torch.int32, device="cuda")
    bt = dinp["block_table"].clone()
    bt[0, 1] = 10 ** 6                                      # sequence 0 loses its second page
    dinp["block_table"] = bt
    got = _run(wl, dinp, 64).numpy()
    status = binding.fa_decode_device_status()
    assert status & binding.FA_STATUS_LEN_CLAMPED
    assert status & binding.FA_STATUS_BAD_BLOCK
    assert np.all(np.isfinite(got))
    assert_close(got[2], want[2], False, "untouched sequence 2")
