#!/usr/bin/env python3
"""Decode-step attention benchmark on GB300: µs per step and KV-read GB/s.

One step = one fa_decode call (split-K kernel + log-sum-exp merge kernel)
over every sequence of the workload, inputs resident in HBM.  The headline
line is measured on the largest decode workload that fits one GPU: 32
sequences of 32K keys, 32 query / 8 KV heads, head_dim 128, paged fp16
K/V (32x32k_d128_paged, 4.29 GB of K/V per step); every decode workload,
that one included, is measured too and listed under "configs".

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier and
torch.cuda.synchronize() on both sides; each step is timed with CUDA events on
the launching stream.  When a workload's KV bytes are under 4x the L2 size,
L2 is flushed before every step outside its events (512 MiB written, then a
read-only pass over another 512 MiB so no dirty lines are left to write
back); larger workloads read more than L2 per step anyway.  The split
kernel's own duration comes from events the library records around it
(fa_decode_profile_next) on the same stream.  Flushed
workloads are also timed with L2 hot (hot_l2: the same steps back to back,
queued behind a GPU sleep so no step waits on the host), beside the cold
headline.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the reference arm of this benchmark).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attention µs/step and KV-read GB/s (fraction of GB300 HBM peak)"
HEADLINE = "32x32k_d128_paged"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--only", action="store_true", help="measure only --workload (for profiling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling only: keep the first N sequences of --workload")
    return ap.parse_args()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None when that summary was taken on a different kernel source
    (the counters then no longer describe the code being timed)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "decode_step_kv_gb300", "csrc", "fa_decode.cu")
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    recorded_sha = recorded = None
    for line in text.splitlines():
        if "source sha256:" in line:
            recorded_sha = line.split("source sha256:")[1].split()[0].strip()
        if "traffic_bytes_per_launch:" in line:
            recorded = int(line.split("traffic_bytes_per_launch:")[1].split()[0])
    return recorded if recorded_sha == sha else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- our arm
def prepare(wl, device):
    import torch
    from decode_step_kv_gb300 import binding
    from decode_step_kv_gb300.inputs import make_inputs
    d = make_inputs(wl, device)
    if wl.v_int8:
        vf = d.pop("v_f32")
        codes = torch.empty(vf.shape, dtype=torch.int8, device=device)
        scales = torch.empty(vf.shape[:-1] + (wl.head_dim // 32,), dtype=torch.float16,
                             device=device)
        binding.fa_quantize_v_int8(vf, codes, scales)
        del vf
        d["v_cache"], d["v_scales"] = codes, scales
    else:
        d["v_scales"] = None
    cap = d["max_blocks"] * (wl.page_size if wl.paged else 1)
    d["workspace"] = binding.alloc_workspace(wl.batch, wl.n_q_heads, wl.n_kv_heads,
                                             wl.head_dim, cap, device=device)
    d["out"] = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), dtype=torch.float32,
                           device=device)
    return d


def call(wl, d, stream, out=None):
    from decode_step_kv_gb300 import binding
    binding.fa_decode(d["q"], d["k_cache"], d["v_cache"], d["v_scales"], d["block_table"],
                      d["seq_lens"], wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.scale,
                      d["window"], d["out"] if out is None else out, batch=wl.batch,
                      page_size=wl.page_size, max_blocks_per_seq=d["max_blocks"],
                      num_blocks=d["num_blocks"] if wl.paged else 0, workspace=d["workspace"],
                      stream=stream)


def l2_note(nbytes):
    """How the timing protocol treats L2 for a step that reads `nbytes`."""
    return ("flushed before every step: 512 MiB written, then 512 MiB read (clean lines)"
            if nbytes < 4 * L2_BYTES else "inputs larger than 4x L2")


def line_config(wl, nbytes, world):
    """The `config` object of a JSON line: the same for both arms."""
    from decode_step_kv_gb300.inputs import WORKLOAD_DESCRIPTIONS
    return {"workload": f"{wl.name}: {WORKLOAD_DESCRIPTIONS[wl.name]}",
            "batch": wl.batch, "n_q_heads": wl.n_q_heads, "n_kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim, "kv_bytes_per_step": nbytes, "l2": l2_note(nbytes),
            "parallelism": f"replicas x{world} (no collectives)"}


class L2Flush:
    """Leave L2 holding none of the step's data between timed steps: write a
    512 MiB buffer (evicts everything) and then reduce over another 512 MiB
    buffer (a read-only pass, so the lines left in L2 are clean and the timed
    kernel never pays to write them back).  Runs outside the timed events.
    Used when a step reads less than 4x L2; larger steps evict L2 by
    themselves."""

    def __init__(self, device):
        import torch
        self.a = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
        self.b = torch.zeros(64 * 2 ** 20, dtype=torch.int64, device=device)

    def __call__(self, i):
        self.a.fill_(i & 0xFF)
        self.b.amax()


def time_kernel(wl, d, steps, warmup, world, device, clocks_gpu=None):
    """Kernel-only timing.  Returns dict with per-step and split-kernel µs."""
    import torch
    from decode_step_kv_gb300 import binding
    from decode_step_kv_gb300.inputs import kv_bytes
    nbytes = kv_bytes(wl, d["lens"], None if d["window"] is None else d["window"].tolist())
    flush = L2Flush(device) if nbytes < 4 * L2_BYTES else None
    stream = torch.cuda.current_stream(device)
    for i in range(warmup):
        if flush:
            flush(i)
        call(wl, d, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    sampler = ClockSampler(clocks_gpu) if clocks_gpu is not None else None
    barrier(world)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.__enter__()
    t0 = time.perf_counter()
    for i in range(steps):
        if flush:
            flush(i)
        ev[i][0].record(stream)
        call(wl, d, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    barrier(world)
    if sampler:
        sampler.__exit__()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # second pass, same steps: the library records an event right after the
    # split kernel (this pass is not the step timing: the event sits between
    # the two kernels and stops the merge from overlapping the split's tail)
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for _, e in ev2:
        e.record(stream)           # creates the CUDA event before the timed steps
    torch.cuda.synchronize(device)
    for i in range(steps):
        if flush:
            flush(i)
        ev2[i][0].record(stream)
        binding.fa_decode_profile_next(None, ev2[i][1])   # recorded after the split kernel
        call(wl, d, stream)
    torch.cuda.synchronize(device)
    split_ms = [a.elapsed_time(b) for a, b in ev2]
    hot_us = None
    if flush:
        # hot L2 (reported beside the cold headline, never instead of it): the
        # same steps back to back with no flush, after one warm call.  A GPU
        # sleep holds the stream while the host queues them all, so no step
        # waits on the host's launch and the events time the GPU alone.
        call(wl, d, stream)
        ev3 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize(device)
        torch.cuda._sleep(int(2e9 * (1e-3 + steps * 50e-6)))
        for i in range(steps):
            ev3[i][0].record(stream)
            call(wl, d, stream)
            ev3[i][1].record(stream)
        torch.cuda.synchronize(device)
        hot_us = 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev3)
    del flush
    res = {
        "hot_us_per_step": hot_us,
        "us_per_step": 1e3 * statistics.mean(step_ms),
        "us_per_step_median": 1e3 * statistics.median(step_ms),
        "split_us": 1e3 * statistics.mean(split_ms),
        "kv_bytes": nbytes,
        "wall_s": wall,
        "l2": l2_note(nbytes),
        "launches": 2 * steps,      # split + merge per timed step
    }
    if sampler:
        res["clocks"] = sampler.summary()
    return res


BI_SPLIT_TOKENS = (256, 1024)   # split sizes the batch-invariant mode is timed at


def time_batch_invariant(wl, d, steps, warmup, device, split_tokens):
    """fa_decode_batch_invariant on the same inputs and with the same cold-L2
    protocol as the headline: µs per step."""
    import torch
    from decode_step_kv_gb300 import binding
    from decode_step_kv_gb300.inputs import kv_bytes
    cap = d["max_blocks"] * (wl.page_size if wl.paged else 1)
    n = binding.fa_decode_batch_invariant_workspace_size(wl.batch, wl.n_q_heads, wl.n_kv_heads,
                                                         wl.head_dim, cap, split_tokens)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device)
    nbytes = kv_bytes(wl, d["lens"], None if d["window"] is None else d["window"].tolist())
    stream = torch.cuda.current_stream(device)

    def step():
        binding.fa_decode_batch_invariant(
            d["q"], d["k_cache"], d["v_cache"], d["v_scales"], d["block_table"], d["seq_lens"],
            wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.scale, d["window"], d["out"],
            split_tokens=split_tokens, batch=wl.batch, page_size=wl.page_size,
            max_blocks_per_seq=d["max_blocks"], num_blocks=d["num_blocks"] if wl.paged else 0,
            workspace=ws, stream=stream)

    return time_steps(step, nbytes, steps, warmup, device)


def time_steps(step, nbytes, steps, warmup, device):
    """Mean µs of `step()` under the headline's protocol: CUDA events on the
    current stream, L2 flushed before every step when it reads under 4x L2."""
    import torch
    flush = L2Flush(device) if nbytes < 4 * L2_BYTES else None
    stream = torch.cuda.current_stream(device)
    for i in range(warmup):
        if flush:
            flush(i)
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize(device)
    for i in range(steps):
        if flush:
            flush(i)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    del flush
    return 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev)


def time_next_rows(steps, device, peak):
    """The rows beyond the plain decode step, each timed under the headline's
    protocol on seeded inputs of the decode shapes: ring-cache decode,
    slot-map decode, multi-query decode, int8 V at head_dim 128, cache
    append."""
    import torch
    from decode_step_kv_gb300 import binding
    from decode_step_kv_gb300.inputs import WORKLOADS, kv_bytes, make_inputs, make_queries
    stream = torch.cuda.current_stream(device)
    res = {}

    # ring cache: 64x128-64k_d128_win's heads and lengths (tokens seen ~U[128, 64K]) on a
    # 4096-row ring per sequence, the storage of a sliding-window layer
    C = 4096
    wl = dataclasses.replace(WORKLOADS["64x128-64k_d128_win"], name="ring", paged=False, window=0,
                             window_odd_only=False)
    d = make_inputs(wl, device, capacity=C)
    B, Hq, Hkv, D = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    nbytes = sum(min(L, C) for L in d["lens"]) * Hkv * D * 4
    ws = binding.alloc_workspace(B, Hq, Hkv, D, C + 16, device=device)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
    us = time_steps(lambda: binding.fa_decode_ring(
        d["q"], d["k_cache"], d["v_cache"], None, d["seq_lens"], Hq, Hkv, D, wl.scale, None, out,
        workspace=ws, stream=stream), nbytes, steps, 3, device)
    gbs = nbytes / (us * 1e-6) / 1e9
    res["ring"] = {"workload": "64 seqs, 32 q/4 kv heads, D=128, 4096-row ring per sequence, "
                               "tokens seen ~U[128, 65536]",
                   "us_per_step": round(us, 2), "kv_bytes": nbytes, "GB/s": round(gbs, 1),
                   "frac_of_peak": round(gbs / peak, 4)}
    del d, ws, out
    torch.cuda.empty_cache()

    # slot map: 8 active slots of a pool of 64 contiguous per-slot caches (32
    # q / 8 kv heads, D=128, 16K keys per slot) through fa_decode_slots, and
    # the same 8 rows decoded the way a caller without the map must: a
    # 64-row fa_decode whose 56 idle rows have length 0
    n_slots, C = 64, 16384
    wl = dataclasses.replace(WORKLOADS["32x32k_d128_paged"], name="slots", batch=n_slots,
                             paged=False, seq_lens=(C,) * n_slots)
    d = make_inputs(wl, device, capacity=C)
    B, Hq, Hkv, D = 8, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    g = torch.Generator(device="cpu").manual_seed(wl.seed + 3000)
    active = torch.randperm(n_slots, generator=g)[:B].to(torch.int32)
    slot_ids = active.to(device)
    lens = torch.full((B,), C, dtype=torch.int32, device=device)
    q8 = d["q"][:B].contiguous()
    nbytes = B * C * Hkv * D * 4
    ws = binding.alloc_workspace(B, Hq, Hkv, D, C, device=device)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
    us = time_steps(lambda: binding.fa_decode_slots(
        q8, d["k_cache"], d["v_cache"], None, slot_ids, lens, Hq, Hkv, D, wl.scale, None, out,
        workspace=ws, stream=stream), nbytes, steps, 3, device)
    q64 = torch.zeros_like(d["q"])
    q64[active.long()] = q8
    lens64 = torch.zeros((n_slots,), dtype=torch.int32)
    lens64[active.long()] = C
    lens64 = lens64.to(device)
    ws64 = binding.alloc_workspace(n_slots, Hq, Hkv, D, C, device=device)
    out64 = torch.empty((n_slots, Hq, D), dtype=torch.float32, device=device)
    us64 = time_steps(lambda: binding.fa_decode(
        q64, d["k_cache"], d["v_cache"], None, None, lens64, Hq, Hkv, D, wl.scale, None, out64,
        batch=n_slots, max_blocks_per_seq=C, workspace=ws64, stream=stream), nbytes, steps, 3,
        device)
    gbs = nbytes / (us * 1e-6) / 1e9
    res["slots_8_of_64"] = {
        "workload": "8 active slots (seeded permutation) of a 64-slot pool of contiguous caches, "
                    "32 q/8 kv heads, D=128, 16384 keys per active slot",
        "us_per_step": round(us, 2), "kv_bytes": nbytes, "GB/s": round(gbs, 1),
        "frac_of_peak": round(gbs / peak, 4),
        "all_64_rows_idle_len0_us_per_step": round(us64, 2)}
    del d, ws, ws64, out, out64, q64
    torch.cuda.empty_cache()

    # multi-query decode (speculative verify) on 32x32k_d128_paged's shape: with G = 4,
    # 2 queries make 8 (query, head) columns per KV head (one column group),
    # 4 queries make 16 (two groups, so each K/V tile is read twice)
    wl = WORKLOADS["32x32k_d128_paged"]
    d = prepare(wl, device)
    B, Hq, Hkv, D = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    nbytes = kv_bytes(wl, d["lens"], None)
    cap = d["max_blocks"] * wl.page_size
    for tq in (2, 4):
        q = make_queries(wl, tq, device)
        n = binding.fa_decode_multi_workspace_size(B, tq, Hq, Hkv, D, cap)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device)
        out = torch.empty((B, tq, Hq, D), dtype=torch.float32, device=device)
        us = time_steps(lambda: binding.fa_decode_multi(
            q, d["k_cache"], d["v_cache"], None, d["block_table"], d["seq_lens"], Hq, Hkv, D,
            wl.scale, None, out, max_blocks_per_seq=d["max_blocks"], num_blocks=d["num_blocks"],
            workspace=ws, stream=stream), nbytes, steps, 3, device)
        gbs = nbytes / (us * 1e-6) / 1e9
        res[f"multi_query_tq{tq}"] = {
            "workload": f"32x32k_d128_paged shape (32 x 32K, 32 q/8 kv heads, D=128, paged), {tq} queries "
                        "per sequence", "us_per_step": round(us, 2), "kv_bytes": nbytes,
            "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "column_groups": -(-tq * wl.group // 8)}
        del ws, out, q

    # multi-query decode at D=256: 16x16k_d256_int8v's shape with fp16 V and 8 queries (16
    # columns per KV head: two groups per warp, the query rows in shared memory)
    wl2 = dataclasses.replace(WORKLOADS["16x16k_d256_int8v"], name="16x16k_d256_fp16v", v_int8=False)
    d2 = prepare(wl2, device)
    B2, Hq2, Hkv2, D2 = wl2.batch, wl2.n_q_heads, wl2.n_kv_heads, wl2.head_dim
    nbytes2 = kv_bytes(wl2, d2["lens"], None)
    q = make_queries(wl2, 8, device)
    n = binding.fa_decode_multi_workspace_size(B2, 8, Hq2, Hkv2, D2,
                                               d2["max_blocks"] * wl2.page_size)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device)
    out = torch.empty((B2, 8, Hq2, D2), dtype=torch.float32, device=device)
    us = time_steps(lambda: binding.fa_decode_multi(
        q, d2["k_cache"], d2["v_cache"], None, d2["block_table"], d2["seq_lens"], Hq2, Hkv2, D2,
        wl2.scale, None, out, max_blocks_per_seq=d2["max_blocks"], num_blocks=d2["num_blocks"],
        workspace=ws, stream=stream), nbytes2, steps, 3, device)
    gbs = nbytes2 / (us * 1e-6) / 1e9
    res["multi_query_d256_tq8"] = {
        "workload": "16 x 16K, 16 q/8 kv heads, D=256, paged, fp16 V (16x16k_d256_int8v with fp16 V), "
                    "8 queries per sequence", "us_per_step": round(us, 2), "kv_bytes": nbytes2,
        "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "column_groups": 2}
    del d2, q, ws, out
    torch.cuda.empty_cache()

    # the same with 16x16k_d256_int8v's own int8 V
    wl3 = WORKLOADS["16x16k_d256_int8v"]
    d3 = prepare(wl3, device)
    nbytes3 = kv_bytes(wl3, d3["lens"], None)
    q = make_queries(wl3, 8, device)
    n = binding.fa_decode_multi_workspace_size(B2, 8, Hq2, Hkv2, D2,
                                               d3["max_blocks"] * wl3.page_size)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device)
    out = torch.empty((B2, 8, Hq2, D2), dtype=torch.float32, device=device)
    us = time_steps(lambda: binding.fa_decode_multi(
        q, d3["k_cache"], d3["v_cache"], d3["v_scales"], d3["block_table"], d3["seq_lens"], Hq2,
        Hkv2, D2, wl3.scale, None, out, max_blocks_per_seq=d3["max_blocks"],
        num_blocks=d3["num_blocks"], workspace=ws, stream=stream), nbytes3, steps, 3, device)
    gbs = nbytes3 / (us * 1e-6) / 1e9
    res["multi_query_d256_int8_tq8"] = {
        "workload": "16x16k_d256_int8v (16 x 16K, 16 q/8 kv heads, D=256, paged, int8 V), "
                    "8 queries per sequence", "us_per_step": round(us, 2), "kv_bytes": nbytes3,
        "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "column_groups": 2}
    del d3, q, ws, out
    torch.cuda.empty_cache()

    # int8 V at head_dim 128: 32x32k_d128_paged's shape with its V packed to int8
    wl4 = dataclasses.replace(WORKLOADS["32x32k_d128_paged"], name="32x32k_d128_paged_int8v",
                              v_int8=True)
    d4 = prepare(wl4, device)
    B4, Hq4, Hkv4, D4 = wl4.batch, wl4.n_q_heads, wl4.n_kv_heads, wl4.head_dim
    nbytes4 = kv_bytes(wl4, d4["lens"], None)
    ws = binding.alloc_workspace(B4, Hq4, Hkv4, D4, d4["max_blocks"] * wl4.page_size,
                                 device=device)
    out = torch.empty((B4, Hq4, D4), dtype=torch.float32, device=device)
    us = time_steps(lambda: binding.fa_decode(
        d4["q"], d4["k_cache"], d4["v_cache"], d4["v_scales"], d4["block_table"], d4["seq_lens"],
        Hq4, Hkv4, D4, wl4.scale, None, out, batch=B4, page_size=wl4.page_size,
        max_blocks_per_seq=d4["max_blocks"], num_blocks=d4["num_blocks"], workspace=ws,
        stream=stream), nbytes4, steps, 3, device)
    gbs = nbytes4 / (us * 1e-6) / 1e9
    res["int8v_d128"] = {
        "workload": "32x32k_d128_paged with int8 V (32 x 32K, 32 q/8 kv heads, D=128, paged)",
        "us_per_step": round(us, 2), "kv_bytes": nbytes4, "GB/s": round(gbs, 1),
        "frac_of_peak": round(gbs / peak, 4)}
    del d4, ws, out
    torch.cuda.empty_cache()

    # cache append: one new K/V row per (sequence, KV head) at each sequence's
    # last position, into 32x32k_d128_paged's paged cache (fp16 V) and 16x16k_d256_int8v's (int8 V)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed + 2000)
    for name, w2 in (("append", wl), ("append_int8", WORKLOADS["16x16k_d256_int8v"])):
        dd = d if w2 is wl else prepare(w2, device)
        B, Hkv, D = w2.batch, w2.n_kv_heads, w2.head_dim
        k_new = torch.randn((B, Hkv, D), generator=g, device=device)
        v_new = torch.randn((B, Hkv, D), generator=g, device=device)
        pos = (dd["seq_lens"] - 1).to(torch.int32)
        row_bytes = B * Hkv * D * (4 + (3 if w2.v_int8 else 2)) + (B * Hkv * (D // 32) * 2
                                                                   if w2.v_int8 else 0)
        us = time_steps(lambda: binding.fa_append_kv(
            k_new, v_new, dd["k_cache"], dd["v_cache"], dd["v_scales"], dd["block_table"], pos,
            n_kv_heads=Hkv, head_dim=D, page_size=w2.page_size,
            max_blocks_per_seq=dd["max_blocks"], num_blocks=dd["num_blocks"], stream=stream),
            row_bytes, steps, 3, device)
        res[name] = {"workload": f"{w2.name} cache: {B} seqs x {Hkv} kv heads x D={D} rows "
                                 f"({'int8' if w2.v_int8 else 'fp16'} V)",
                     "us_per_call": round(us, 2)}
        if dd is not d:
            del dd
    del d
    torch.cuda.empty_cache()
    return res


def e2e_copies(wl, lens, host, dev):
    """The host->device copies of one end-to-end step, as (destination,
    source) pairs.  A contiguous cache ([B][Hkv][cap][...]) crosses as each
    (sequence, KV head)'s written rows [0, L_b), which are contiguous on both
    sides, not its whole capacity; a paged cache crosses as its whole block
    pool; every other input whole."""
    copies = []
    for n, src in host.items():
        if not wl.paged and n in ("k_cache", "v_cache", "v_scales"):
            for b, L in enumerate(lens):
                for kv in range(wl.n_kv_heads):
                    if L > 0:
                        copies.append((dev[n][b, kv, :L], src[b, kv, :L]))
        else:
            copies.append((dev[n], src))
    return copies


def time_e2e(wl, d, steps, warmup, device):
    """Same step through the public API with host inputs: pinned host -> device
    copies of the step's inputs (e2e_copies), fa_decode, device -> host copy of
    the output.  Also reports whether that output is bit-identical to the
    resident step's."""
    import torch
    names = ["q", "k_cache", "v_cache", "v_scales", "block_table", "seq_lens", "window"]
    host = {n: d[n].cpu().pin_memory() for n in names if d.get(n) is not None}
    dev = {n: torch.empty_like(d[n]) for n in host}
    copies = e2e_copies(wl, d["lens"], host, dev)
    out_h = torch.empty(d["out"].shape, dtype=torch.float32).pin_memory()
    h2d = sum(src.numel() * src.element_size() for _, src in copies)
    d2h = out_h.numel() * 4
    stream = torch.cuda.current_stream(device)
    dd = dict(d)
    dd["out"] = torch.empty_like(d["out"])

    def step():
        for dst, src in copies:
            dst.copy_(src, non_blocking=True)
        dd.update(dev)
        call(wl, dd, stream)
        out_h.copy_(dd["out"], non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    call(wl, d, stream)                       # the resident step, same plan
    torch.cuda.synchronize(device)
    same = bool(torch.equal(out_h, d["out"].cpu()))
    return ms, h2d, d2h, same


def time_e2e_serving(wl, d, steps, warmup, device):
    """A serving decode step through the public API, cache resident on the
    device: copy this step's q and new K/V rows (and positions) from pinned
    host memory, append the rows with fa_append_kv at each sequence's last
    position, run fa_decode, copy the output back."""
    import torch
    from decode_step_kv_gb300 import binding
    B, Hkv, D = wl.batch, wl.n_kv_heads, wl.head_dim
    g = torch.Generator().manual_seed(wl.seed + 77)
    parts = {
        "q": d["q"].cpu(),
        "k_new": torch.randn((B, Hkv, D), generator=g),
        "v_new": torch.randn((B, Hkv, D), generator=g),
        "pos": torch.tensor([L - 1 for L in d["lens"]], dtype=torch.int32),
    }
    # the step's inputs packed in one pinned buffer (16-byte aligned parts),
    # so they cross to the device in one copy, as a server would send them
    offs, total = {}, 0
    for k, t in parts.items():
        offs[k] = total
        total += -(-t.numel() * t.element_size() // 16) * 16
    host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=device)
    dev = {}
    for k, t in parts.items():
        nb = t.numel() * t.element_size()
        host_buf[offs[k]:offs[k] + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
        dev[k] = dev_buf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    out_h = torch.empty(d["out"].shape, dtype=torch.float32).pin_memory()
    h2d = total
    stream = torch.cuda.current_stream(device)
    dd = dict(d)

    def step():
        dev_buf.copy_(host_buf, non_blocking=True)
        binding.fa_append_kv(dev["k_new"], dev["v_new"], d["k_cache"], d["v_cache"],
                             d.get("v_scales"), d["block_table"], dev["pos"],
                             n_kv_heads=Hkv, head_dim=D, page_size=wl.page_size,
                             max_blocks_per_seq=d["max_blocks"],
                             num_blocks=d["num_blocks"] if wl.paged else 0)
        dd["q"] = dev["q"]
        call(wl, dd, stream)
        out_h.copy_(dd["out"], non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return ms, h2d, out_h.numel() * 4


# --------------------------------------------------------------- CPU oracle
def oracle_sample(wl, inp, budget_s, threads=0):
    """Time the oracle on whole (sequence, kv-head) units of the workload until
    about `budget_s` of CPU work; returns (GB/s, seconds, units, threads)."""
    import oracle
    from decode_step_kv_gb300.inputs import attended_tokens
    lens = inp["lens"]
    win = None if inp["window"] is None else inp["window"].tolist()
    toks = attended_tokens(lens, win)
    G = wl.group
    vrow = wl.head_dim * (1 if wl.v_int8 else 2) + (wl.head_dim // 32 * 2 if wl.v_int8 else 0)
    unit_bytes = [t * (2 * wl.head_dim + vrow) for t in toks]
    n_threads = threads if threads > 0 else (os.cpu_count() or 1)
    n_units = wl.batch * wl.n_kv_heads
    per_call = max(1, -(-n_threads // G))       # enough rows to keep every core busy
    done_bytes, elapsed, units, start, used = 0, 0.0, 0, 0, 1
    while elapsed < budget_s:
        chunk = [(start + i) % n_units for i in range(per_call)]
        start += per_call
        rows = []
        for u in chunk:
            b, kv = divmod(u, wl.n_kv_heads)
            rows += [b * wl.n_q_heads + kv * G + g for g in range(G)]
        used = max(used, min(n_threads, len(rows)))
        t0 = time.perf_counter()
        oracle.decode(inp["q"].numpy(), inp["k_cache"].numpy(), inp["v_cache"].numpy(), lens,
                      scale=wl.scale, n_kv_heads=wl.n_kv_heads,
                      v_scales=None if inp.get("v_scales") is None else inp["v_scales"].numpy(),
                      block_table=None if inp["block_table"] is None
                      else inp["block_table"].numpy(),
                      window=None if inp["window"] is None else inp["window"].numpy(),
                      page_size=wl.page_size, max_blocks=inp["max_blocks"], rows=rows,
                      threads=n_threads)
        elapsed += time.perf_counter() - t0
        done_bytes += sum(unit_bytes[u // wl.n_kv_heads] for u in chunk)
        units += len(chunk)
    return done_bytes / elapsed / 1e9, elapsed, units, used


def cpu_inputs(wl):
    import torch
    from decode_step_kv_gb300.inputs import make_inputs
    inp = make_inputs(wl, "cpu")
    if wl.v_int8:
        import oracle
        c, s = oracle.pack_v_int8(inp.pop("v_f32").numpy())
        inp["v_cache"] = torch.from_numpy(c)
        inp["v_scales"] = torch.from_numpy(s.copy())
    else:
        inp["v_scales"] = None
    return inp


# --------------------------------------------------------------- arms
def run_ours(args, world, rank, local):
    import torch
    from decode_step_kv_gb300 import binding
    from decode_step_kv_gb300.inputs import WORKLOADS, WORKLOAD_DESCRIPTIONS
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    binding.load()
    peak, peak_kind = measured_peaks()
    wl = WORKLOADS[args.workload]
    if args.batch:
        wl = dataclasses.replace(wl, batch=args.batch, seq_lens=None if wl.seq_lens is None
                                 else wl.seq_lens[:args.batch])
    d = prepare(wl, device)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    r = time_kernel(wl, d, args.steps, args.warmup, world, device, clocks_gpu=gpu_index)
    us = max_over_ranks(r["us_per_step"], world)
    split_us = max_over_ranks(r["split_us"], world)
    gbs_total = world * r["kv_bytes"] / (us * 1e-6) / 1e9
    achieved = r["kv_bytes"] / (split_us * 1e-6) / 1e9
    kernel = ("fa_split_kernel" if os.environ.get("FA_DECODE_KERNEL") == "simt"
              else "fa_stream_mma_kernel")
    traffic = recorded_traffic(kernel, wl.name) if not args.batch else None
    line = {
        "metric": METRIC,
        "value": round(gbs_total, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 6),
        "us_per_step": round(us, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "math": ("fp16 x fp16 products on the tensor cores (mma.sync), fp32 accumulation and "
                 "softmax; P rounded to fp16 for the PV product; fp16 K/V"
                 + (", int8 V x fp16 scale" if wl.v_int8 else "")),
        "data": "synthetic (seeded N(0,1) fp16 q/K/V, random block tables)",
        "config": line_config(wl, r["kv_bytes"], world),
        "frac_of_hbm_peak": round(gbs_total / world / peak, 4),
        "roofline": {"bound": "hbm", "kernel": kernel,
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "peak_kind": peak_kind, "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": r["kv_bytes"]},
        "gpu_launches": r["launches"],
        "clocks": r.get("clocks"),
    }
    if r["hot_us_per_step"] is not None:
        hot = max_over_ranks(r["hot_us_per_step"], world)
        line["hot_l2"] = {"us_per_step": round(hot, 2),
                          "value": round(r["kv_bytes"] / (hot * 1e-6) / 1e9 * world, 2),
                          "unit": "GB/s",
                          "note": "same steps back to back without the L2 flush (informative; "
                                  "the headline is cold L2)"}
    if not args.no_e2e:
        ms, h2d, d2h, same = time_e2e(wl, d, max(5, args.steps // 5), 2, device)
        line["e2e"] = {"value": round(r["kv_bytes"] / (ms * 1e-3) / 1e9 * world, 2),
                       "unit": "GB/s", "us_per_step": round(ms * 1e3, 2),
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "output_equals_resident": same,
                       "note": "every input copied host->device each step: a contiguous "
                               "cache as each (sequence, kv head)'s written rows, a paged "
                               "cache as its whole block pool"}
        ms2, h2d2, d2h2 = time_e2e_serving(wl, d, max(5, args.steps // 5), 2, device)
        line["e2e_serving"] = {"value": round(r["kv_bytes"] / (ms2 * 1e-3) / 1e9 * world, 2),
                               "unit": "GB/s", "us_per_step": round(ms2 * 1e3, 2),
                               "h2d_bytes_per_step": h2d2, "d2h_bytes_per_step": d2h2,
                               "note": "cache resident; per step: q, the new K/V rows and "
                                       "their positions host->device in one copy, "
                                       "fa_append_kv, fa_decode, out device->host"}
    del d
    torch.cuda.empty_cache()
    if not args.only:
        per = {}
        for name, other in WORKLOADS.items():
            dd = prepare(other, device)
            rr = time_kernel(other, dd, max(10, min(args.steps, 30)), 3, world, device)
            gbs = rr["kv_bytes"] / (rr["us_per_step"] * 1e-6) / 1e9
            per[name] = {"us_per_step": round(rr["us_per_step"], 2),
                         "split_us": round(rr["split_us"], 2),
                         "kv_bytes": rr["kv_bytes"], "GB/s": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4),
                         "split_frac_of_peak": round(rr["kv_bytes"] / (rr["split_us"] * 1e-6)
                                                     / 1e9 / peak, 4),
                         "l2": rr["l2"]}
            if rr["hot_us_per_step"] is not None:
                per[name]["hot_l2_us_per_step"] = round(rr["hot_us_per_step"], 2)
            per[name]["batch_invariant_us_per_step"] = {
                str(st): round(time_batch_invariant(other, dd, max(10, min(args.steps, 30)), 3,
                                                    device, st), 2)
                for st in BI_SPLIT_TOKENS}
            del dd
            torch.cuda.empty_cache()
        line["configs"] = per
        line["next_rows"] = time_next_rows(max(10, min(args.steps, 30)), device, peak)
        line["batch_invariant"] = {
            "split_tokens": list(BI_SPLIT_TOKENS),
            "note": "each workload entry's batch_invariant_us_per_step[split_tokens]: "
                    "fa_decode_batch_invariant on the same inputs and protocol (fixed splits "
                    "per sequence, bit-identical whatever the batch)"}
    if rank == 0 and world == 1 and not args.no_cpu:
        inp = cpu_inputs(wl)
        gbs, secs, units, thr = oracle_sample(wl, inp, budget_s=12.0)
        gbs1, secs1, units1, _ = oracle_sample(wl, inp, budget_s=3.0, threads=1)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": thr,
                                "kind": "oracle",
                                "sample": f"{units} (sequence, kv-head) units of {wl.name}, "
                                          f"all query heads of each, {secs:.1f} s",
                                "one_core_value": round(gbs1, 4),
                                "one_core_sample": f"{units1} units on one thread, {secs1:.1f} s"}
    if rank == 0:
        print(json.dumps(line))


def run_reference(args, world, rank):
    """The fp64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    from decode_step_kv_gb300.inputs import WORKLOADS, kv_bytes
    wl = WORKLOADS[args.workload]
    inp = cpu_inputs(wl)
    # the K/V bytes of the workload's step (its lengths are fixed, or drawn
    # with the inputs)
    lens = inp.get("lens") or list(wl.seq_lens or ())
    win = inp.get("window")
    nbytes = kv_bytes(wl, lens, None if win is None else win.tolist())
    per_step_budget = max(0.2, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(wl, inp, budget_s=per_step_budget)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        gbs, s, units, thr = oracle_sample(wl, inp, budget_s=per_step_budget)
        vals.append(gbs)
        secs += s
    v = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(wl, nbytes, world),
            "cpu_baseline": {"kind": "oracle", "cores": thr, "value": round(v, 4),
                             "unit": "GB/s",
                             "sample": f"per step: whole (sequence, kv-head) units of {wl.name} "
                                       f"for ~{per_step_budget:.1f} s"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
