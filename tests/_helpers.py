"""Shared plumbing for the GPU parity tests: inputs, calls, error metrics."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload, make_inputs

FP16_NAN = 0x7E00

# Tolerances: max abs error 2e-3 (fp16 cache) / 1e-2 (int8 V), relative L2 <= 1e-3.
TOL = {False: (2e-3, 1e-3), True: (1e-2, 1e-3)}


def poison_unused(inp, wl: Workload):
    """Fill every cache row outside [0, L_b) (and spare blocks) with NaN, so a
    kernel that reads or weights an unattended row fails the comparison."""
    P = wl.page_size
    keys = ["k_cache", "v_cache"] if "v_cache" in inp else ["k_cache"]
    for key in keys:
        c = inp[key]
        u16 = c.view(torch.int16)
        if wl.paged:
            used = torch.zeros(c.shape[0], dtype=torch.bool)
            bt = inp["block_table"].cpu()
            for b, L in enumerate(inp["lens"]):
                nb = -(-L // P)
                used[bt[b, :nb].long()] = True
                if L % P and nb:
                    u16[int(bt[b, nb - 1]), :, L % P:] = FP16_NAN
            u16[~used.to(c.device)] = FP16_NAN
        else:
            for b, L in enumerate(inp["lens"]):
                u16[b, :, L:] = FP16_NAN
    return inp


def pack_on_cpu(inp):
    """int8 V through the oracle's packer (the oracle side's V)."""
    codes, scales = oracle.pack_v_int8(inp["v_f32"].cpu().numpy())
    return torch.from_numpy(codes), torch.from_numpy(scales.view(np.float16).copy())


def build_case(wl: Workload, *, seq_lens=None, capacity=None, spare_blocks=0, poison=True):
    inp = make_inputs(wl, "cpu", seq_lens=seq_lens, capacity=capacity, spare_blocks=spare_blocks)
    if wl.v_int8:
        codes, scales = pack_on_cpu(inp)
        inp["v_cache"], inp["v_scales"] = codes, scales
        if poison:
            sc = inp["v_scales"].view(torch.int16)
            P = wl.page_size
            if wl.paged:
                bt = inp["block_table"]
                for b, L in enumerate(inp["lens"]):
                    nb = -(-L // P)
                    if L % P and nb:
                        sc[int(bt[b, nb - 1]), :, L % P:] = FP16_NAN
            else:
                for b, L in enumerate(inp["lens"]):
                    sc[b, :, L:] = FP16_NAN
    else:
        inp["v_scales"] = None
    if poison:
        poison_unused(inp, wl)
    return inp


def to_cuda(inp):
    out = {}
    for k, v in inp.items():
        out[k] = v.cuda() if isinstance(v, torch.Tensor) else v
    return out


def gpu_decode(wl: Workload, dinp, *, stream=None, poison_ws=True, out=None):
    B, Hq, Hkv, D = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    cap = dinp["max_blocks"] * (wl.page_size if wl.paged else 1)
    ws = binding.alloc_workspace(B, Hq, Hkv, D, cap)
    if poison_ws:
        ws.view(torch.uint8).fill_(0xFF)   # NaN pattern for every float in the scratch
    if out is None:
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    binding.fa_decode(dinp["q"], dinp["k_cache"], dinp["v_cache"], dinp.get("v_scales"),
                      dinp["block_table"], dinp["seq_lens"], Hq, Hkv, D, wl.scale,
                      dinp["window"], out, batch=B, page_size=wl.page_size,
                      max_blocks_per_seq=dinp["max_blocks"],
                      num_blocks=dinp["num_blocks"] if wl.paged else 0, workspace=ws,
                      stream=stream)
    return out


def oracle_decode(wl: Workload, inp, rows=None, threads=0):
    return oracle.decode(inp["q"].numpy(), inp["k_cache"].numpy(), inp["v_cache"].numpy(),
                         inp["lens"], scale=wl.scale, n_kv_heads=wl.n_kv_heads,
                         v_scales=None if inp.get("v_scales") is None else inp["v_scales"].numpy(),
                         block_table=None if inp["block_table"] is None
                         else inp["block_table"].numpy(),
                         window=None if inp["window"] is None else inp["window"].numpy(),
                         page_size=wl.page_size, max_blocks=inp["max_blocks"], rows=rows,
                         threads=threads)


def errors(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = got - want
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(want))
    rel_l2 = float(np.linalg.norm(diff)) / den if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel_l2


def assert_close(got, want, int8: bool, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel = errors(got, want)
    tol_abs, tol_rel = TOL[int8]
    assert max_abs <= tol_abs and rel <= tol_rel, (
        f"{what}: max abs {max_abs:.3e} (tol {tol_abs}), rel L2 {rel:.3e} (tol {tol_rel})")
    return max_abs, rel
