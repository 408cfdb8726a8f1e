"""Seeded synthetic inputs for decode-step attention.

This module only draws random numbers and lays them out; it holds none of the
attention or quantisation arithmetic.  The tests (and the CPU oracle they
drive) and the benchmark both take their inputs from here, so both sides see
identical bytes.

Recipe (the same for every workload):
  * one torch.Generator, seed = 20261202 + workload index (CPU for small cases,
    CUDA for the full-size ones, so the two streams differ but each is fixed);
  * q, K and V drawn N(0, 1) in fp32 and rounded to fp16 (round to nearest);
    for the int8-V cache the fp32 V draw is returned for the caller to pack;
  * paged caches: 16-token pages; physical block ids are a seeded random
    permutation of all blocks the sequences need, sliced per sequence in order;
    unused block-table entries hold -1;
  * ragged lengths: either listed or drawn uniform in [lo, hi] by randint.

The five named workloads are the decode shapes the method is measured on:
  1x512_d128  1 seq, 8 q / 2 kv heads, D 128, L 512, contiguous fp16
  4x1k-8k_d256  4 seqs, 16 q / 8 kv heads, D 256, L {1024, 2048, 4096, 8192}, contiguous
  32x32k_d128_paged  32 seqs, 32 q / 8 kv heads, D 128, L 32768, paged (split-K long context)
  16x16k_d256_int8v  16 seqs, 16 q / 8 kv heads, D 256, L 16384, paged, K fp16 + V int8
  64x128-64k_d128_win  64 seqs, 32 q / 4 kv heads, D 128, L ~ U[128, 65536], paged,
        sliding window 4096 on odd-indexed sequences
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    seq_lens: Optional[Sequence[int]] = None      # listed lengths, or
    len_range: Optional[tuple] = None             # (lo, hi) drawn uniform, inclusive
    paged: bool = False
    page_size: int = 16
    v_int8: bool = False
    window: int = 0                               # window size, 0 = none
    window_odd_only: bool = False                 # window only on odd-indexed sequences
    seed: int = BASE_SEED

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    "1x512_d128": Workload("1x512_d128", 1, 8, 2, 128, seq_lens=(512,), seed=BASE_SEED + 0),
    "4x1k-8k_d256": Workload("4x1k-8k_d256", 4, 16, 8, 256, seq_lens=(1024, 2048, 4096, 8192),
                     seed=BASE_SEED + 1),
    "32x32k_d128_paged": Workload("32x32k_d128_paged", 32, 32, 8, 128, seq_lens=(32768,) * 32, paged=True,
                     seed=BASE_SEED + 2),
    "16x16k_d256_int8v": Workload("16x16k_d256_int8v", 16, 16, 8, 256, seq_lens=(16384,) * 16, paged=True,
                     v_int8=True, seed=BASE_SEED + 3),
    "64x128-64k_d128_win": Workload("64x128-64k_d128_win", 64, 32, 4, 128, len_range=(128, 65536), paged=True,
                     window=4096, window_odd_only=True, seed=BASE_SEED + 4),
}

WORKLOAD_DESCRIPTIONS = {
    "1x512_d128": "1 seq, 8 q/2 kv heads, D=128, L=512, contiguous fp16 K/V",
    "4x1k-8k_d256": "4 seqs, 16 q/8 kv heads, D=256, L={1024,2048,4096,8192}, contiguous fp16 K/V",
    "32x32k_d128_paged": "32 seqs, 32 q/8 kv heads, D=128, L=32768, paged 16-token pages, fp16 K/V",
    "16x16k_d256_int8v": "16 seqs, 16 q/8 kv heads, D=256, L=16384, paged, fp16 K + int8 V (fp16 scale/32)",
    "64x128-64k_d128_win": "64 seqs, 32 q/4 kv heads, D=128, L~U[128,65536], paged, window 4096 on odd seqs",
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_lengths(wl: Workload, g: torch.Generator) -> list:
    if wl.seq_lens is not None:
        return [int(x) for x in wl.seq_lens]
    lo, hi = wl.len_range
    # drawn on the CPU generator stream order regardless of device
    return [int(x) for x in torch.randint(lo, hi + 1, (wl.batch,), generator=g,
                                          device=g.device).tolist()]


def _normal_fp16(shape, g, device, chunk_elems=1 << 28):
    """N(0,1) drawn in fp32 and rounded to fp16, in chunks along dim 0."""
    out = torch.empty(shape, dtype=torch.float16, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    rows = max(1, chunk_elems // max(1, flat.shape[1]))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                  dtype=torch.float32).to(torch.float16)
    return out


def _normal_fp32(shape, g, device, chunk_elems=1 << 28):
    out = torch.empty(shape, dtype=torch.float32, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    rows = max(1, chunk_elems // max(1, flat.shape[1]))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                  dtype=torch.float32)
    return out


def make_inputs(wl: Workload, device="cpu", *, seq_lens: Optional[Sequence[int]] = None,
                capacity: Optional[int] = None, spare_blocks: int = 0):
    """Draw one batch of inputs for `wl` on `device`.

    Returns a dict with q [B,Hq,D] fp16, k_cache fp16, v_cache (fp16) or
    v_f32 (fp32 draw, int8 workloads: the caller packs it), block_table
    [B,max_blocks] int32 or None, seq_lens [B] int32, window [B] int32 or None,
    max_blocks (blocks per sequence, or capacity in tokens when contiguous),
    num_blocks, page_size, and the host-side list `lens`.
    `capacity` (tokens) overrides the per-sequence capacity; `spare_blocks`
    adds unused physical blocks to the paged pool.
    """
    device = torch.device(device)
    g = _gen(wl.seed, device)
    lens = list(seq_lens) if seq_lens is not None else draw_lengths(wl, g)
    B, Hq, Hkv, D, P = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size
    assert len(lens) == B
    cap = capacity if capacity is not None else max(max(lens), 1)
    if wl.paged:
        cap = -(-cap // P) * P
    q = _normal_fp16((B, Hq, D), g, device)
    out = {"q": q, "lens": lens, "page_size": P}
    if wl.paged:
        per_seq = [-(-L // P) for L in lens]
        max_blocks = cap // P
        total = sum(per_seq) + spare_blocks
        perm = torch.randperm(total, generator=g, device=device).to(torch.int32)
        bt = torch.full((B, max_blocks), -1, dtype=torch.int32, device=device)
        off = 0
        for b, n in enumerate(per_seq):
            bt[b, :n] = perm[off:off + n]
            off += n
        kv_shape = (total, Hkv, P, D)
        out.update(block_table=bt, max_blocks=max_blocks, num_blocks=total)
    else:
        kv_shape = (B, Hkv, cap, D)
        out.update(block_table=None, max_blocks=cap, num_blocks=0)
    out["k_cache"] = _normal_fp16(kv_shape, g, device)
    if wl.v_int8:
        out["v_f32"] = _normal_fp32(kv_shape, g, device)
    else:
        out["v_cache"] = _normal_fp16(kv_shape, g, device)
    out["seq_lens"] = torch.tensor(lens, dtype=torch.int32, device=device)
    if wl.window > 0:
        w = [wl.window if (not wl.window_odd_only or b % 2 == 1) else 0 for b in range(B)]
        out["window"] = torch.tensor(w, dtype=torch.int32, device=device)
    else:
        out["window"] = None
    return out


def make_queries(wl: Workload, n_queries: int, device="cpu"):
    """q [B, n_queries, Hq, D] fp16 for multi-query decode: N(0,1) rounded to
    fp16 from its own seeded stream (seed + 1000)."""
    g = _gen(wl.seed + 1000, torch.device(device))
    return _normal_fp16((wl.batch, n_queries, wl.n_q_heads, wl.head_dim), g, torch.device(device))


def attended_tokens(lens, window) -> list:
    """Per-sequence number of keys in the attended range (window applied)."""
    res = []
    for b, L in enumerate(lens):
        W = 0 if window is None else int(window[b])
        res.append(min(L, W) if W > 0 else L)
    return res


def kv_bytes(wl: Workload, lens, window) -> int:
    """Algorithmic K + V (+ scale) bytes one decode step must read."""
    toks = sum(attended_tokens(lens, window)) * wl.n_kv_heads
    k = toks * wl.head_dim * 2
    if wl.v_int8:
        v = toks * wl.head_dim + toks * (wl.head_dim // 32) * 2
    else:
        v = toks * wl.head_dim * 2
    return k + v
