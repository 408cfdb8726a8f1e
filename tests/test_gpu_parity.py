"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases compare every output element; the full-size decode workloads
compare sampled (sequence, head) rows the oracle computes one by one, in the
launch configuration the benchmark times.  Unattended cache rows are NaN and
the workspace starts as NaN, so reading or weighting either shows up.
"""
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import WORKLOADS, Workload, make_inputs

from _helpers import (assert_close, build_case, gpu_decode, oracle_decode, to_cuda)

pytestmark = pytest.mark.gpu


def W(name, B, Hq, Hkv, D, **kw):
    return Workload(name, B, Hq, Hkv, D, seed=7000 + zlib.crc32(name.encode()) % 1000, **kw)


SMALL = [
    # (workload, explicit lengths)
    (W("d128_g4_contig", 6, 8, 2, 128), [1, 15, 16, 17, 100, 700]),
    (W("d128_g4_paged", 6, 8, 2, 128, paged=True), [1, 15, 16, 17, 100, 700]),
    (W("d256_g2_contig", 6, 4, 2, 256), [1, 7, 8, 9, 333, 1500]),
    (W("d256_g2_paged", 6, 4, 2, 256, paged=True), [1, 7, 8, 9, 333, 1500]),
    (W("d128_g1", 3, 2, 2, 128, paged=True), [5, 64, 1000]),
    (W("d128_g2", 3, 4, 2, 128), [5, 64, 1000]),
    (W("d128_g8_groups", 3, 16, 2, 128, paged=True), [5, 64, 1000]),
    (W("d128_g3_padded", 3, 6, 2, 128), [5, 64, 1000]),
    (W("d256_g1", 3, 2, 2, 256, paged=True), [5, 64, 1000]),
    (W("d256_g16_groups", 2, 16, 1, 256, paged=True), [77, 600]),
    (W("d128_window", 4, 8, 2, 128, paged=True, window=40), [100, 1000, 1000, 37]),
    (W("d256_window_odd", 4, 4, 2, 256, window=256, window_odd_only=True), [100, 1000, 1000, 37]),
    (W("d128_empty_rows", 4, 8, 2, 128, paged=True), [0, 33, 0, 1]),
    (W("d128_int8_paged", 4, 8, 2, 128, paged=True, v_int8=True), [1, 17, 300, 1025]),
    (W("d256_int8_paged", 4, 4, 2, 256, paged=True, v_int8=True), [1, 9, 300, 1025]),
    (W("d256_int8_contig", 3, 4, 2, 256, v_int8=True), [3, 200, 511]),
    (W("d128_int8_window", 3, 8, 2, 128, paged=True, v_int8=True, window=100), [50, 500, 333]),
    (W("d128_page64", 3, 8, 2, 128, paged=True, page_size=64), [63, 64, 1000]),
    # many short ragged sequences (with empty ones): work ranges cross unit
    # boundaries and units cross work ranges
    (W("d128_many_ragged", 40, 8, 2, 128, paged=True),
     [(i * 37) % 211 if i % 7 else 0 for i in range(40)]),
    (W("d256_many_ragged_int8", 33, 8, 4, 256, paged=True, v_int8=True),
     [(i * 53) % 301 if i % 5 else 0 for i in range(33)]),
    (W("d128_g16_long", 2, 32, 2, 128, paged=True), [20000, 9]),
    # the largest GQA group accepted (64 query heads on one KV head) and the
    # narrowest window (only the newest token)
    (W("d128_g64", 2, 64, 1, 128, paged=True), [3000, 77]),
    (W("d256_window1", 3, 4, 2, 256, paged=True, window=1), [1, 2, 999]),
]


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


@pytest.mark.parametrize("wl,lens", SMALL, ids=[w.name for w, _ in SMALL])
def test_small_cases_match_oracle(wl, lens, kernel):
    cap = max(lens)
    if wl.v_int8 and not wl.paged:
        cap = -(-cap // 16) * 16
    inp = build_case(wl, seq_lens=lens, capacity=cap, spare_blocks=3 if wl.paged else 0)
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, wl.v_int8, wl.name)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0)


def test_run_to_run_bit_identical(kernel):
    wl = W("det", 4, 8, 2, 128, paged=True)
    inp = to_cuda(build_case(wl, seq_lens=[100, 2000, 3000, 17], spare_blocks=2))
    a = gpu_decode(wl, inp).cpu()
    b = gpu_decode(wl, inp).cpu()
    assert torch.equal(a, b)


def test_batched_equals_one_sequence_at_a_time(kernel):
    """A multi-sequence call equals single-sequence calls (within tolerance;
    the split plans differ, so bitwise equality is not required)."""
    wl = W("batched", 4, 8, 2, 128, paged=True)
    lens = [100, 2000, 3000, 17]
    inp = build_case(wl, seq_lens=lens)
    dinp = to_cuda(inp)
    whole = gpu_decode(wl, dinp).cpu().numpy()
    wl1 = dataclasses.replace(wl, batch=1)
    for b in range(4):
        one = dict(dinp)
        one["q"] = dinp["q"][b:b + 1].contiguous()
        one["block_table"] = dinp["block_table"][b:b + 1].contiguous()
        one["seq_lens"] = dinp["seq_lens"][b:b + 1].contiguous()
        got = gpu_decode(wl1, one).cpu().numpy()
        assert_close(got[0], whole[b], False, f"seq {b}")


def test_non_default_stream():
    wl = W("stream", 2, 8, 2, 128, paged=True)
    inp = build_case(wl, seq_lens=[700, 1500])
    want = oracle_decode(wl, inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dinp = to_cuda(inp)
        got = gpu_decode(wl, dinp, stream=s)
    s.synchronize()
    assert_close(got.cpu().numpy(), want, False, "stream")


def test_length_beyond_capacity_is_clamped_and_flagged(kernel):
    wl = W("clamp", 2, 8, 2, 128, paged=True)
    inp = build_case(wl, seq_lens=[64, 32])
    binding.fa_decode_device_status()                       # clear
    dinp = to_cuda(inp)
    dinp["seq_lens"] = torch.tensor([64, 10 ** 6], dtype=torch.int32, device="cuda")
    got = gpu_decode(wl, dinp).cpu().numpy()
    status = binding.fa_decode_device_status()
    assert status & binding.FA_STATUS_LEN_CLAMPED
    # capacity of sequence 1 is max_blocks * 16 = 64 tokens (its pages 2, 3 are
    # unassigned (-1) and flagged as bad blocks, so only its first 32 count)
    assert status & binding.FA_STATUS_BAD_BLOCK
    want = oracle_decode(wl, inp)
    assert_close(got[0], want[0], False, "clamped seq 0")
    assert_close(got[1], want[1], False, "clamped seq 1 (only its 32 stored keys)")


def test_bad_block_id_is_skipped_and_flagged(kernel):
    wl = W("badblk", 2, 8, 2, 128, paged=True)
    inp = build_case(wl, seq_lens=[64, 64])
    dinp = to_cuda(inp)
    binding.fa_decode_device_status()
    bt = dinp["block_table"].clone()
    bt[1, 2] = 10 ** 6                                      # out of range: tile skipped
    dinp["block_table"] = bt
    got = gpu_decode(wl, dinp).cpu().numpy()
    assert binding.fa_decode_device_status() & binding.FA_STATUS_BAD_BLOCK
    want = oracle_decode(wl, inp)
    assert_close(got[0], want[0], False, "untouched seq 0")
    assert np.all(np.isfinite(got[1]))


@pytest.mark.parametrize("what", ["k", "v16", "v8", "scales"])
def test_gather_bit_exact(what):
    P = 16
    wl = W("gather", 3, 8, 2, 256 if what in ("v8", "scales") else 128, paged=True,
           v_int8=what in ("v8", "scales"))
    lens = [45, 16, 300]
    inp = build_case(wl, seq_lens=lens, poison=False, spare_blocks=4)
    cache = {"k": inp["k_cache"], "v16": inp["v_cache"], "v8": inp["v_cache"],
             "scales": inp["v_scales"]}[what]
    row_bytes = int(np.prod(cache.shape[3:])) * cache.element_size()
    dcache = cache.cuda()
    dbt = inp["block_table"].cuda()
    for b, L in enumerate(lens):
        dense = torch.zeros((wl.n_kv_heads, L) + tuple(cache.shape[3:]), dtype=cache.dtype,
                            device="cuda")
        binding.fa_gather_kv_debug(dcache, row_bytes, dbt, b, wl.n_kv_heads, P,
                                   inp["max_blocks"], inp["num_blocks"], L, dense)
        want = oracle.gather_rows(cache.numpy(), inp["block_table"].numpy(), b, L,
                                  n_kv_heads=wl.n_kv_heads, page_size=P)
        got = dense.cpu().numpy()
        assert got.tobytes() == want.tobytes()


@pytest.mark.parametrize("D", [128, 256])
def test_gpu_packer_bit_exact(D):
    g = torch.Generator().manual_seed(D)
    x = torch.randn((517, D), generator=g)
    x[3] *= 1e-9                                            # scale underflows to 0
    x[4] = 0
    x[5, :32] = torch.tensor([127.0, -63.5, 0.5, 1.5, -2.5, 2.5, 126.4, -127.0] + [0.0] * 24)
    want_c, want_s = oracle.pack_v_int8(x.numpy())
    dx = x.cuda()
    codes = torch.empty((517, D), dtype=torch.int8, device="cuda")
    scales = torch.empty((517, D // 32), dtype=torch.float16, device="cuda")
    binding.fa_quantize_v_int8(dx, codes, scales)
    assert codes.cpu().numpy().tobytes() == want_c.tobytes()
    assert scales.cpu().numpy().view(np.uint16).tobytes() == want_s.view(np.uint16).tobytes()


# ------------------------------------------------------------- full-size cases
def _sampled_rows(wl, lens, n_seq=4, seed=0):
    rng = np.random.default_rng(seed)
    seqs = sorted(set([0, wl.batch - 1] + list(rng.choice(wl.batch, n_seq, replace=False))))
    rows = []
    for b in seqs:
        for h in sorted(set([0, wl.n_q_heads - 1, int(rng.integers(wl.n_q_heads))])):
            rows.append(b * wl.n_q_heads + h)
    return rows


def _oracle_rows_paged(wl, dinp, rows, v_codes=None, v_scales=None):
    """Oracle on the sampled rows: each sampled sequence's blocks are copied to
    the host (a compact paged cache, identity block table)."""
    res = {}
    P = wl.page_size
    by_seq = {}
    for r in rows:
        by_seq.setdefault(r // wl.n_q_heads, []).append(r % wl.n_q_heads)
    for b, heads in by_seq.items():
        L = dinp["lens"][b]
        nb = -(-L // P)
        sel = dinp["block_table"][b, :nb].long()
        k = dinp["k_cache"].index_select(0, sel).cpu().numpy()
        if wl.v_int8:
            v = v_codes(sel)
            sc = v_scales(sel)
        else:
            v = dinp["v_cache"].index_select(0, sel).cpu().numpy()
            sc = None
        bt = np.arange(nb, dtype=np.int32)[None, :]
        win = None if dinp["window"] is None else [int(dinp["window"][b])]
        q = dinp["q"][b:b + 1].cpu().numpy()
        out = oracle.decode(q, k, v, [L], scale=wl.scale, n_kv_heads=wl.n_kv_heads,
                            v_scales=sc, block_table=bt, window=win, page_size=P,
                            max_blocks=nb, rows=heads)
        for i, h in enumerate(heads):
            res[b * wl.n_q_heads + h] = out[i]
    return res


@pytest.mark.parametrize("name", ["1x512_d128", "4x1k-8k_d256"])
def test_small_workloads_full_oracle(name, kernel):
    wl = WORKLOADS[name]
    inp = build_case(wl)
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, wl.v_int8, name)


@pytest.mark.parametrize("name", ["32x32k_d128_paged", "16x16k_d256_int8v", "64x128-64k_d128_win"])
def test_full_size_workloads_sampled(name):
    wl = WORKLOADS[name]
    torch.cuda.empty_cache()
    dinp = make_inputs(wl, "cuda")
    if wl.v_int8:
        vf = dinp.pop("v_f32")
        codes = torch.empty(vf.shape, dtype=torch.int8, device="cuda")
        scales = torch.empty(vf.shape[:-1] + (wl.head_dim // 32,), dtype=torch.float16,
                             device="cuda")
        binding.fa_quantize_v_int8(vf, codes, scales)
        dinp["v_cache"], dinp["v_scales"] = codes, scales

        def v_codes(sel):
            c, _ = oracle.pack_v_int8(vf.index_select(0, sel).cpu().numpy())
            # the GPU packer must agree bit for bit with the oracle's packer
            assert c.tobytes() == codes.index_select(0, sel).cpu().numpy().tobytes()
            return c

        def v_scales(sel):
            _, s = oracle.pack_v_int8(vf.index_select(0, sel).cpu().numpy())
            assert (s.view(np.uint16).tobytes()
                    == scales.index_select(0, sel).cpu().numpy().view(np.uint16).tobytes())
            return s
    else:
        dinp["v_scales"] = None
        v_codes = v_scales = None
    got = gpu_decode(wl, dinp).cpu().numpy().reshape(wl.batch * wl.n_q_heads, wl.head_dim)
    rows = _sampled_rows(wl, dinp["lens"])
    want = _oracle_rows_paged(wl, dinp, rows, v_codes, v_scales)
    g = np.stack([got[r] for r in rows])
    w = np.stack([want[r] for r in rows])
    assert_close(g, w, wl.v_int8, name)
    assert np.all(np.isfinite(got))
    del dinp
    torch.cuda.empty_cache()


def test_many_sequences_take_the_general_length_scan():
    """More than 128 sequences: the kernels' two-pass scan over the lengths
    (the one-pass register scan covers up to 128)."""
    B = 300
    lens = [(i * 37) % 97 + (0 if i % 11 else 0) for i in range(B)]
    lens[5] = 0
    lens[250] = 2000
    wl = W("many_seqs", B, 8, 2, 128, paged=True, window=50, window_odd_only=True)
    inp = build_case(wl, seq_lens=lens, spare_blocks=3)
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, False, "300 sequences")


@pytest.mark.parametrize("D,int8", [(128, False), (256, False), (256, True)])
def test_many_rows_take_the_warp_per_row_merge(D, int8):
    """48 sequences x 16 query heads = 768 output rows, at or above four rows
    per SM: the merge runs a warp per row, eight rows per CTA."""
    B = 48
    lens = [(i * 211) % 3000 + (0 if i % 13 else 0) for i in range(B)]
    lens[3] = 0
    wl = W(f"many_rows_{D}_{int(int8)}", B, 16, 4, D, paged=True, v_int8=int8, window=700,
           window_odd_only=True)
    inp = build_case(wl, seq_lens=lens, spare_blocks=2)
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, int8, wl.name)
    assert np.all(got[3] == 0)


@pytest.mark.parametrize("D,Hq,int8", [(128, 32, False), (128, 32, True), (256, 32, False)])
def test_sixteen_query_heads_per_kv_head_take_two_column_groups(D, Hq, int8):
    """G = 16 with a block table of 2^20 tokens per sequence: the K/V the
    capacity allows passes the two-group threshold, so a warp carries 16
    columns (at D=256 with the query rows in shared memory)."""
    wl = W(f"two_groups_{D}_{int(int8)}", 3, Hq, 2, D, paged=True, v_int8=int8, window=500,
           window_odd_only=True)
    lens = [20000, 9, 1700]
    inp = build_case(wl, seq_lens=lens, capacity=1 << 20, spare_blocks=2)
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, int8, wl.name)


def test_one_long_unit_spans_every_worker():
    """One sequence, one KV head, one query head: the unit's partials come
    from every worker of the grid, so the merge folds more than 512 slots in
    several passes."""
    wl = W("one_unit", 1, 1, 1, 128, paged=True)
    inp = build_case(wl, seq_lens=[40000])
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, False, "one long unit")


def test_batch_beyond_the_register_scan_publishes_the_prefix():
    """More than 256 sequences: the split kernel's worker 0 publishes the
    per-sequence prefix that the merge kernel reads instead of rescanning."""
    B = 600
    lens = [(i * 53) % 131 for i in range(B)]
    lens[7] = 3000
    wl = W("prefix_published", B, 8, 2, 128, paged=True)
    inp = build_case(wl, seq_lens=lens, spare_blocks=2)
    want = oracle_decode(wl, inp)
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, want, False, "600 sequences")
