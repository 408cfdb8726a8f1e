"""Seeded random sweep of the decode entry points against the oracle.

Each case draws a shape (head_dim, KV heads, group size, batch), ragged
lengths (empty sequences included), windows, the cache layout (paged or
contiguous, fp16 or int8 V) and an entry point: fa_decode, fa_decode_multi,
fa_decode_ring and their batch-invariant forms.  Paged cases take pages of
16, 32 or 64 tokens; a quarter of the single-query fa_decode and
fa_decode_ring cases run on the CUDA-core split kernel (FA_DECODE_KERNEL=simt)
instead of the tensor-core one, and about a third of the rest hold the
tensor-core kernel to the stream-K plan (FA_DECODE_PLAN=streamk) where the
library would take the cluster plan of small steps.  A paged case outside the batch-invariant
forms may take a block table of 2^20 tokens per sequence, which moves the
planner to 16-column units when a KV head has more than 8 columns; batches of
many rows reach the warp-per-row merge.  Unwritten cache rows and the
workspace hold NaN, so a read or weight of either shows up.
"""
import contextlib
import os
import zlib

import numpy as np
import pytest
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, to_cuda

pytestmark = pytest.mark.gpu

MODES = ["decode", "multi", "ring", "decode_bi", "multi_bi", "ring_bi"]
N_CASES = int(os.environ.get("FA_FUZZ_CASES", "150"))   # more seeds for a longer sweep


def _draw(seed):
    r = np.random.default_rng(9900 + seed)
    mode = MODES[seed % len(MODES)]
    D = int(r.choice([128, 256]))
    Hkv = int(r.choice([1, 2, 4]))
    G = int(r.choice([1, 2, 3, 4, 8, 16, 4, 8]))
    B = int(r.integers(1, 13))
    if r.random() < 0.15:
        B = int(r.integers(40, 80))                      # many rows: warp-per-row merge
    Lmax = int(r.choice([40, 300, 3000]))
    lens = [int(x) if r.random() > 0.1 else 0 for x in r.integers(1, Lmax + 1, B)]
    window = int(r.choice([0, 0, 1, 17, 200]))
    int8 = bool(r.random() < 0.35)
    paged = bool(r.random() < 0.6)
    # a 2^20-token block table only matters for 16-column units, which the
    # batch-invariant plan never uses (and whose scratch grows with capacity
    # over split size)
    big_cap = paged and not mode.endswith("_bi") and bool(r.random() < 0.6)
    tq = int(r.integers(2, 7)) if mode.startswith("multi") else 1
    split = int(r.choice([16, 64, 256, 512]))
    P = int(r.choice([16, 16, 32, 64])) if paged else 16
    simt = mode in ("decode", "ring") and bool(r.random() < 0.25)
    # the tensor-core kernel held to the stream-K plan in some cases that the
    # library would give the cluster plan (drawn last: earlier draws unchanged)
    streamk = bool(r.random() < 0.3)
    return dict(mode=mode, D=D, Hkv=Hkv, G=G, B=B, lens=lens, window=window, int8=int8,
                paged=paged, big_cap=big_cap, tq=tq, split=split, P=P, simt=simt,
                streamk=streamk, seed=seed)


def _ws(n):
    return torch.full((max(int(n), 16),), 0xFF, dtype=torch.uint8, device="cuda")


def _run_paged_or_contig(c):
    mode, D, Hkv, G, B, tq = c["mode"], c["D"], c["Hkv"], c["G"], c["B"], c["tq"]
    Hq = G * Hkv
    name = f"fuzz{c['seed']}"
    wl = Workload(name, B, Hq, Hkv, D, paged=c["paged"], page_size=c["P"], v_int8=c["int8"],
                  window=c["window"], window_odd_only=c["seed"] % 2 == 1,
                  seed=20000 + zlib.crc32(name.encode()) % 1000)
    cap = max(max(c["lens"]), 1)
    if c["big_cap"]:
        cap = 1 << 20
    if not c["paged"]:
        cap = -(-cap // 16) * 16
    inp = build_case(wl, seq_lens=c["lens"], capacity=cap, spare_blocks=2 if c["paged"] else 0)
    d = to_cuda(inp)
    cap_tok = d["max_blocks"] * (c["P"] if c["paged"] else 1)
    kw = dict(max_blocks_per_seq=d["max_blocks"], num_blocks=d["num_blocks"] if c["paged"] else 0,
              page_size=c["P"])
    okw = dict(scale=wl.scale, n_kv_heads=Hkv,
               v_scales=None if not c["int8"] else inp["v_scales"].numpy(),
               block_table=None if not c["paged"] else inp["block_table"].numpy(),
               window=None if inp["window"] is None else inp["window"].numpy(), page_size=c["P"],
               max_blocks=inp["max_blocks"])
    if mode in ("decode", "decode_bi"):
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        if mode == "decode":
            ws = binding.alloc_workspace(B, Hq, Hkv, D, cap_tok)
            ws.fill_(0xFF)
            binding.fa_decode(d["q"], d["k_cache"], d["v_cache"], d.get("v_scales"),
                              d["block_table"], d["seq_lens"], Hq, Hkv, D, wl.scale, d["window"],
                              out, workspace=ws, **kw)
        else:
            ws = _ws(binding.fa_decode_batch_invariant_workspace_size(B, Hq, Hkv, D, cap_tok,
                                                                      c["split"]))
            binding.fa_decode_batch_invariant(d["q"], d["k_cache"], d["v_cache"],
                                              d.get("v_scales"), d["block_table"], d["seq_lens"],
                                              Hq, Hkv, D, wl.scale, d["window"], out,
                                              split_tokens=c["split"], workspace=ws, **kw)
        want = oracle.decode(inp["q"].numpy(), inp["k_cache"].numpy(), inp["v_cache"].numpy(),
                             c["lens"], **okw)
    else:
        q = np.random.default_rng(c["seed"]).standard_normal((B, tq, Hq, D)).astype(np.float16)
        qd = torch.from_numpy(q).cuda()
        out = torch.full((B, tq, Hq, D), float("nan"), device="cuda")
        if mode == "multi":
            ws = _ws(binding.fa_decode_multi_workspace_size(B, tq, Hq, Hkv, D, cap_tok))
            binding.fa_decode_multi(qd, d["k_cache"], d["v_cache"], d.get("v_scales"),
                                    d["block_table"], d["seq_lens"], Hq, Hkv, D, wl.scale,
                                    d["window"], out, workspace=ws, **kw)
        else:
            ws = _ws(binding.fa_decode_multi_batch_invariant_workspace_size(
                B, tq, Hq, Hkv, D, cap_tok, c["split"]))
            binding.fa_decode_multi_batch_invariant(qd, d["k_cache"], d["v_cache"],
                                                    d.get("v_scales"), d["block_table"],
                                                    d["seq_lens"], Hq, Hkv, D, wl.scale,
                                                    d["window"], out, split_tokens=c["split"],
                                                    workspace=ws, **kw)
        want = oracle.decode_multi(q, inp["k_cache"].numpy(), inp["v_cache"].numpy(), c["lens"],
                                   **okw)
    return out.cpu().numpy(), want


def _run_ring(c):
    D, Hkv, G, B = c["D"], c["Hkv"], c["G"], c["B"]
    Hq = G * Hkv
    r = np.random.default_rng(30000 + c["seed"])
    C = int(r.choice([32, 64, 128]))
    seen = [int(x) for x in r.integers(1, 4 * C + 1, B)]
    q = r.standard_normal((B, Hq, D)).astype(np.float16)
    k = r.standard_normal((B, Hkv, C, D)).astype(np.float16)
    if c["int8"]:
        v, sc = oracle.pack_v_int8(r.standard_normal((B, Hkv, C, D)).astype(np.float32))
    else:
        v, sc = r.standard_normal((B, Hkv, C, D)).astype(np.float16), None
    for b, n in enumerate(seen):                   # rows never written yet
        if n < C:
            k[b, :, n:] = np.nan
            if sc is None:
                v[b, :, n:] = np.nan
            else:
                sc[b, :, n:] = np.nan
    win = np.array([c["window"]] * B, dtype=np.int32)
    scale = D ** -0.5
    want = oracle.decode_ring(q, k, v, seen, scale=scale, n_kv_heads=Hkv, v_scales=sc, window=win)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    if c["mode"] == "ring":
        ws = _ws(binding.fa_decode_workspace_size(B, Hq, Hkv, D, C + 16))
        binding.fa_decode_ring(t(q), t(k), t(v), t(sc), t(np.array(seen, dtype=np.int32)), Hq,
                               Hkv, D, scale, t(win), out, workspace=ws)
    else:
        ws = _ws(binding.fa_decode_batch_invariant_workspace_size(B, Hq, Hkv, D, C + 16,
                                                                  c["split"]))
        binding.fa_decode_ring_batch_invariant(t(q), t(k), t(v), t(sc),
                                               t(np.array(seen, dtype=np.int32)), Hq, Hkv, D,
                                               scale, t(win), out, split_tokens=c["split"],
                                               workspace=ws)
    return out.cpu().numpy(), want


@contextlib.contextmanager
def _split_kernel(simt, streamk=False):
    """The library reads FA_DECODE_KERNEL and FA_DECODE_PLAN at every call."""
    old = {k: os.environ.get(k) for k in ("FA_DECODE_KERNEL", "FA_DECODE_PLAN")}
    os.environ.pop("FA_DECODE_KERNEL", None)
    os.environ.pop("FA_DECODE_PLAN", None)
    if simt:
        os.environ["FA_DECODE_KERNEL"] = "simt"
    if streamk:
        os.environ["FA_DECODE_PLAN"] = "streamk"
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case_matches_oracle(seed):
    c = _draw(seed)
    with _split_kernel(c["simt"], c["streamk"]):
        got, want = (_run_ring if c["mode"].startswith("ring") else _run_paged_or_contig)(c)
    assert_close(got, want, c["int8"], str(c))
