"""Parity at the sizes the benchmark times for the rows beyond the plain
decode step: multi-query decode (4 queries) and the batch-invariant plan on
the 32 x 32K, 32/8-head, D=128 paged workload, ring decode on 64 sequences
with 64x128-64k_d128_win's heads and lengths over 4096-row rings, the slot
map over a pool of 64 contiguous 16K caches, int8 V at head_dim 128 on the
32 x 32K workload, and 8-query decode on 16x16k_d256_int8v.  The oracle
recomputes a sample of the sequences (every output row of each), each from a
host copy of that sequence's cache alone.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import WORKLOADS, make_inputs, make_queries

from _helpers import assert_close

pytestmark = pytest.mark.gpu


def _sample(B, n=4, seed=0):
    rng = np.random.default_rng(seed)
    return sorted(set([0, B - 1] + [int(x) for x in rng.choice(B, n, replace=False)]))


def _seq_blocks(d, b, P):
    """Sequence b's K/V blocks on the host, with an identity block table."""
    L = d["lens"][b]
    nb = -(-L // P)
    sel = d["block_table"][b, :nb].long()
    k = d["k_cache"].index_select(0, sel).cpu().numpy()
    v = d["v_cache"].index_select(0, sel).cpu().numpy()
    return L, nb, k, v, np.arange(nb, dtype=np.int32)[None, :]


@pytest.fixture(scope="module")
def long_context():
    wl = WORKLOADS["32x32k_d128_paged"]
    torch.cuda.empty_cache()
    d = make_inputs(wl, "cuda")
    yield wl, d
    del d
    torch.cuda.empty_cache()


def test_multi_query_four_queries_at_full_size(long_context):
    """16 (query, head) columns per KV head: the two-column-group kernel."""
    wl, d = long_context
    tq = 4
    B, Hq, Hkv, D = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    q = make_queries(wl, tq, "cuda")
    cap = d["max_blocks"] * wl.page_size
    n = binding.fa_decode_multi_workspace_size(B, tq, Hq, Hkv, D, cap)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, tq, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_multi(q, d["k_cache"], d["v_cache"], None, d["block_table"],
                            d["seq_lens"], Hq, Hkv, D, wl.scale, None, out,
                            max_blocks_per_seq=d["max_blocks"], num_blocks=d["num_blocks"],
                            workspace=ws)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in _sample(B, n=2):
        L, nb, k, v, bt = _seq_blocks(d, b, wl.page_size)
        want = oracle.decode_multi(q[b:b + 1].cpu().numpy(), k, v, [L], scale=wl.scale,
                                   n_kv_heads=Hkv, block_table=bt, page_size=wl.page_size,
                                   max_blocks=nb)
        assert_close(got[b:b + 1], want, False, f"multi-query sequence {b}")


def test_batch_invariant_1024_at_full_size(long_context):
    wl, d = long_context
    B, Hq, Hkv, D = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    cap = d["max_blocks"] * wl.page_size
    n = binding.fa_decode_batch_invariant_workspace_size(B, Hq, Hkv, D, cap, 1024)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_batch_invariant(d["q"], d["k_cache"], d["v_cache"], None,
                                      d["block_table"], d["seq_lens"], Hq, Hkv, D, wl.scale, None,
                                      out, split_tokens=1024, workspace=ws)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in _sample(B, n=2, seed=1):
        L, nb, k, v, bt = _seq_blocks(d, b, wl.page_size)
        want = oracle.decode(d["q"][b:b + 1].cpu().numpy(), k, v, [L], scale=wl.scale,
                             n_kv_heads=Hkv, block_table=bt, page_size=wl.page_size,
                             max_blocks=nb)
        assert_close(got[b:b + 1], want, False, f"batch-invariant sequence {b}")


def test_ring_decode_at_bench_size():
    C = 4096
    wl = dataclasses.replace(WORKLOADS["64x128-64k_d128_win"], name="ring", paged=False, window=0,
                             window_odd_only=False)
    torch.cuda.empty_cache()
    d = make_inputs(wl, "cuda", capacity=C)
    B, Hq, Hkv, D = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    ws = binding.alloc_workspace(B, Hq, Hkv, D, C + 16)
    ws.fill_(0xFF)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_ring(d["q"], d["k_cache"], d["v_cache"], None, d["seq_lens"], Hq, Hkv, D,
                           wl.scale, None, out, workspace=ws)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in _sample(B, n=4, seed=2):
        want = oracle.decode_ring(d["q"][b:b + 1].cpu().numpy(),
                                  d["k_cache"][b:b + 1].cpu().numpy(),
                                  d["v_cache"][b:b + 1].cpu().numpy(), [d["lens"][b]],
                                  scale=wl.scale, n_kv_heads=Hkv)
        assert_close(got[b:b + 1], want, False, f"ring sequence {b} ({d['lens'][b]} tokens)")
    del d
    torch.cuda.empty_cache()


def test_slot_map_eight_of_sixty_four_at_full_size():
    """The benchmark's slot-map row: 8 active slots (a seeded permutation) of a
    64-slot pool of contiguous 16K caches, 32 q / 8 kv heads, D=128.  The
    oracle decodes each sampled row from a host copy of its slot alone (a
    slot map equals the gathered sub-batch)."""
    n_slots, C = 64, 16384
    wl = dataclasses.replace(WORKLOADS["32x32k_d128_paged"], name="slots", batch=n_slots,
                             paged=False, seq_lens=(C,) * n_slots)
    torch.cuda.empty_cache()
    d = make_inputs(wl, "cuda", capacity=C)
    B, Hq, Hkv, D = 8, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    g = torch.Generator(device="cpu").manual_seed(wl.seed + 3000)
    active = torch.randperm(n_slots, generator=g)[:B].to(torch.int32)
    lens = [C, C - 1, 1, 5000, C, 77, 12345, C]          # ragged within the slots' caches
    q8 = d["q"][:B].contiguous()
    ws = torch.full((max(binding.fa_decode_workspace_size(B, Hq, Hkv, D, C), 16),), 0xFF,
                    dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_slots(q8, d["k_cache"], d["v_cache"], None, active.cuda(),
                            torch.tensor(lens, dtype=torch.int32, device="cuda"), Hq, Hkv, D,
                            wl.scale, None, out, workspace=ws)
    got = out.cpu().numpy()
    for b in _sample(B):
        s, L = int(active[b]), lens[b]
        k = d["k_cache"][s:s + 1, :, :L].contiguous().cpu().numpy()
        v = d["v_cache"][s:s + 1, :, :L].contiguous().cpu().numpy()
        want = oracle.decode(q8[b:b + 1].cpu().numpy(), k, v, [L], scale=wl.scale,
                             n_kv_heads=Hkv)
        assert_close(got[b:b + 1], want, False, f"slot {s} (row {b}, {L} keys)")
    assert np.all(np.isfinite(got))
    del d
    torch.cuda.empty_cache()


def test_int8_v_head_dim_128_at_full_size():
    """The benchmark's int8-V head_dim-128 row: 32x32k_d128_paged's shape with
    its V packed to int8 on the GPU (3 CTAs x 4 warps per SM).  Each sampled
    sequence's V blocks are packed again by the oracle's packer from the same
    fp32 draw (the bytes must agree), then decoded by the oracle."""
    wl = dataclasses.replace(WORKLOADS["32x32k_d128_paged"], name="int8v_d128", v_int8=True)
    torch.cuda.empty_cache()
    d = make_inputs(wl, "cuda")
    vf = d.pop("v_f32")
    codes = torch.empty(vf.shape, dtype=torch.int8, device="cuda")
    scales = torch.empty(vf.shape[:-1] + (wl.head_dim // 32,), dtype=torch.float16,
                         device="cuda")
    binding.fa_quantize_v_int8(vf, codes, scales)
    B, Hq, Hkv, D, P = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size
    cap = d["max_blocks"] * P
    ws = torch.full((max(binding.fa_decode_workspace_size(B, Hq, Hkv, D, cap), 16),), 0xFF,
                    dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    binding.fa_decode(d["q"], d["k_cache"], codes, scales, d["block_table"], d["seq_lens"], Hq,
                      Hkv, D, wl.scale, None, out, batch=B, page_size=P,
                      max_blocks_per_seq=d["max_blocks"], num_blocks=d["num_blocks"],
                      workspace=ws)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in _sample(B, n=2, seed=3):
        L = d["lens"][b]
        nb = -(-L // P)
        sel = d["block_table"][b, :nb].long()
        vc, vs = oracle.pack_v_int8(vf.index_select(0, sel).cpu().numpy())
        assert np.array_equal(codes.index_select(0, sel).cpu().numpy(), vc)
        assert np.array_equal(scales.index_select(0, sel).cpu().numpy().view(np.uint16),
                              vs.view(np.uint16))
        want = oracle.decode(d["q"][b:b + 1].cpu().numpy(),
                             d["k_cache"].index_select(0, sel).cpu().numpy(), vc, [L],
                             scale=wl.scale, n_kv_heads=Hkv, v_scales=vs,
                             block_table=np.arange(nb, dtype=np.int32)[None, :], page_size=P,
                             max_blocks=nb)
        assert_close(got[b:b + 1], want, True, f"int8 V sequence {b}")
    del d, vf, codes, scales
    torch.cuda.empty_cache()


def test_multi_query_eight_queries_int8_v_at_full_size():
    """The benchmark's int8-V multi-query row: 16x16k_d256_int8v with 8
    queries per sequence (16 columns per KV head: two column groups per warp
    at head_dim 256, 6 warps per CTA), V packed on the GPU and checked
    against the oracle's packer for the sampled sequences."""
    wl = WORKLOADS["16x16k_d256_int8v"]
    torch.cuda.empty_cache()
    d = make_inputs(wl, "cuda")
    vf = d.pop("v_f32")
    codes = torch.empty(vf.shape, dtype=torch.int8, device="cuda")
    scales = torch.empty(vf.shape[:-1] + (wl.head_dim // 32,), dtype=torch.float16,
                         device="cuda")
    binding.fa_quantize_v_int8(vf, codes, scales)
    tq = 8
    B, Hq, Hkv, D, P = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size
    q = make_queries(wl, tq, "cuda")
    cap = d["max_blocks"] * P
    n = binding.fa_decode_multi_workspace_size(B, tq, Hq, Hkv, D, cap)
    ws = torch.full((max(n, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((B, tq, Hq, D), float("nan"), device="cuda")
    binding.fa_decode_multi(q, d["k_cache"], codes, scales, d["block_table"], d["seq_lens"], Hq,
                            Hkv, D, wl.scale, None, out, max_blocks_per_seq=d["max_blocks"],
                            num_blocks=d["num_blocks"], workspace=ws)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in _sample(B, n=1, seed=4):
        L = d["lens"][b]
        nb = -(-L // P)
        sel = d["block_table"][b, :nb].long()
        vc, vs = oracle.pack_v_int8(vf.index_select(0, sel).cpu().numpy())
        assert np.array_equal(codes.index_select(0, sel).cpu().numpy(), vc)
        want = oracle.decode_multi(q[b:b + 1].cpu().numpy(),
                                   d["k_cache"].index_select(0, sel).cpu().numpy(), vc, [L],
                                   scale=wl.scale, n_kv_heads=Hkv, v_scales=vs,
                                   block_table=np.arange(nb, dtype=np.int32)[None, :],
                                   page_size=P, max_blocks=nb)
        assert_close(got[b:b + 1], want, True, f"int8 V multi-query sequence {b}")
    del d, vf, codes, scales
    torch.cuda.empty_cache()
