"""Host-side checks of the C-ABI library (no GPU needed).

The library loads, exports every entry point include/fa_decode.h declares,
and rejects bad arguments with the documented codes before touching the GPU.
"""
import ctypes
import os
import re

import pytest

from decode_step_kv_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"FA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("fa_decode", "fa_decode_workspace_size"):
        assert required in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_built_for_sm_103a_only():
    text = open(_build.__file__).read()
    assert "arch=compute_103a,code=sm_103a" in text
    assert "sm_90" not in text and "sm_100" not in text


# ------------------------------------------------------------------ validation
A = 1 << 20  # fake, 16-byte aligned "device" addresses: never dereferenced


def call(lib, **kw):
    args = dict(q=A, k=2 * A, v=3 * A, vs=None, bt=None, sl=4 * A, hq=8, hkv=2, d=128,
                scale=0.088, win=None, out=5 * A, batch=1, page=16, maxb=512, nblk=0,
                ws=6 * A, wsb=1 << 30, stream=None)
    args.update(kw)
    rc = lib.fa_decode(args["q"], args["k"], args["v"], args["vs"], args["bt"], args["sl"],
                       args["hq"], args["hkv"], args["d"], args["scale"], args["win"],
                       args["out"], args["batch"], args["page"], args["maxb"], args["nblk"],
                       args["ws"], args["wsb"], args["stream"])
    return rc, lib.fa_decode_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1), (dict(sl=None), -1),
    (dict(out=None), -1),
    (dict(d=64), -2), (dict(d=192), -2),
    (dict(hq=6, hkv=4), -3), (dict(hkv=0), -3), (dict(hq=0), -3), (dict(hq=130, hkv=2), -3),
    (dict(scale=float("inf")), -5), (dict(scale=float("nan")), -5),
    (dict(batch=-1), -6), (dict(maxb=0), -6),
    (dict(bt=7 * A, page=8, nblk=10), -6), (dict(bt=7 * A, page=24, nblk=10), -6),
    (dict(bt=7 * A, page=16, nblk=0), -6),
    (dict(vs=8 * A, maxb=500), -6),                      # contiguous int8 needs cap % 16 == 0
    (dict(q=A + 8), -9), (dict(out=5 * A + 4), -9), (dict(k=2 * A + 2), -9),
    (dict(sl=4 * A + 2), -9), (dict(win=8 * A + 1), -9),            # int32 arrays: 4-byte
    (dict(bt=7 * A + 2, page=16, nblk=10), -9),
    (dict(out=2 * A + 64), -7),                          # out inside the K cache
    (dict(out=A), -7),                                   # out == q
])
def test_bad_arguments_rejected_before_any_launch(lib, kw, code):
    rc, msg = call(lib, **kw)
    assert rc == code, msg
    assert msg


def test_workspace_size_host_only(lib):
    f = lib.fa_decode_workspace_size
    assert f(1, 8, 2, 100, 512, 152) == 0                  # bad head_dim
    assert f(1, 6, 4, 128, 512, 152) == 0                  # heads not divisible
    small = f(1, 8, 2, 128, 512, 152)
    big = f(32, 32, 8, 128, 32768, 152)
    # at least one partial record (D floats of O plus (m, l)) per query head
    assert small >= 8 * (128 * 4 + 8)
    assert big >= 32 * 32 * (128 * 4 + 8)
    assert f(1, 8, 2, 256, 512, 152) > small
    assert big > small > 0
    # more SMs -> at least as many splits
    assert f(32, 32, 8, 128, 32768, 304) >= big
    assert f(0, 8, 2, 128, 512, 152) == 0


def test_quantize_and_gather_reject_bad_arguments(lib):
    assert lib.fa_quantize_v_int8(None, 1, 32, A, A, None) == -1
    assert lib.fa_quantize_v_int8(A, 1, 48, A, A, None) == -2
    assert lib.fa_gather_kv_debug(A, 256, None, 0, 2, 16, 64, 0, 65, A, None) == -6
    assert lib.fa_gather_kv_debug(A, 256, A, 0, 2, 8, 64, 4, 16, A, None) == -6
    assert lib.fa_gather_kv_debug(None, 256, None, 0, 2, 16, 64, 0, 16, A, None) == -1
    assert lib.fa_gather_kv_debug(A, 256, 5 * A + 2, 0, 2, 16, 64, 4, 16, 6 * A, None) == -9
    assert lib.fa_quantize_v_int8(A + 2, 1, 32, 2 * A, 3 * A, None) == -9
    assert lib.fa_quantize_v_int8(A, 1, 32, 2 * A, 3 * A + 1, None) == -9


def test_append_rejects_bad_arguments(lib):
    f = lib.fa_append_kv
    #        k_new v_new k_cache v_cache scales bt  pos  B  Hkv D   P   maxb nblk stream
    assert f(None, A, 2 * A, 3 * A, None, None, 4 * A, 1, 2, 128, 16, 64, 0, None) == -1
    assert f(A, A, 2 * A, 3 * A, None, None, None, 1, 2, 128, 16, 64, 0, None) == -1
    assert f(A, A, 2 * A, 3 * A, None, None, 4 * A, 1, 2, 100, 16, 64, 0, None) == -2
    assert f(A, A, 2 * A, 3 * A, None, None, 4 * A, 1, 0, 128, 16, 64, 0, None) == -3
    assert f(A, A, 2 * A, 3 * A, None, 5 * A, 4 * A, 1, 2, 128, 8, 64, 4, None) == -6
    assert f(A, A, 2 * A, 3 * A, None, None, 4 * A, 1, 2, 128, 16, 0, 0, None) == -6
    # the K cache (1 x 2 x 64 x 128 fp16 = 32 KiB from 2A) would overlap k_new at 2A + 4096
    assert f(2 * A + 4096, A, 2 * A, 3 * A, None, None, 4 * A, 1, 2, 128, 16, 64, 0, None) == -7
    assert f(A, A, 2 * A, 3 * A, None, None, 4 * A, 0, 2, 128, 16, 64, 0, None) == 0   # no-op
    # pointers aligned to their element type: fp32 and int32 4 bytes, fp16 2
    assert f(A + 2, A, 2 * A, 3 * A, None, None, 4 * A, 1, 2, 128, 16, 64, 0, None) == -9
    assert f(A, A, 2 * A + 1, 3 * A, None, None, 4 * A, 1, 2, 128, 16, 64, 0, None) == -9
    assert f(A, A, 2 * A, 3 * A + 1, None, None, 4 * A, 1, 2, 128, 16, 64, 0, None) == -9
    assert f(A, A, 2 * A, 3 * A, 8 * A + 1, None, 4 * A, 1, 2, 128, 16, 64, 0, None) == -9
    assert f(A, A, 2 * A, 3 * A, None, None, 4 * A + 2, 1, 2, 128, 16, 64, 0, None) == -9
    assert f(A, A, 2 * A, 3 * A, None, 5 * A + 2, 4 * A, 1, 2, 128, 16, 64, 4, None) == -9
    g = lib.fa_append_kv_ring
    #        k_new  v_new  k_cache  v_cache scales pos    B  Hkv D    cap stream
    assert g(A, A + 1, 2 * A, 3 * A, None, 4 * A, 1, 2, 128, 64, None) == -9


def test_ring_rejects_bad_capacity(lib):
    f = lib.fa_decode_ring
    #        q  k      v      vs    sl     hq hkv d    scale win  out    B  cap  ws     wsb    st
    assert f(A, 2 * A, 3 * A, None, 4 * A, 8, 2, 128, 0.1, None, 5 * A, 1, 100, 6 * A, 1 << 30,
             None) == -6
    assert f(A, 2 * A, 3 * A, None, 4 * A, 8, 2, 128, 0.1, None, 5 * A, 1, 0, 6 * A, 1 << 30,
             None) == -6
    assert f(A, 2 * A, 3 * A, None, None, 8, 2, 128, 0.1, None, 5 * A, 1, 64, 6 * A, 1 << 30,
             None) == -1
    g = lib.fa_append_kv_ring
    assert g(A, A, 2 * A, 3 * A, None, 4 * A, 1, 2, 128, 100, None) == -6
    assert g(A, A, 2 * A, 3 * A, None, None, 1, 2, 128, 64, None) == -1


def test_multi_rejects_bad_query_count_and_sizes_its_workspace(lib):
    f = lib.fa_decode_multi
    args = lambda tq: (A, 2 * A, 3 * A, None, None, 4 * A, tq, 8, 2, 128, 0.1, None, 5 * A, 1,
                       16, 512, 0, 6 * A, 1 << 30, None)
    assert f(*args(0)) == -6
    assert f(*args(257)) == -6
    g = lib.fa_decode_multi_workspace_size
    assert g(1, 0, 8, 2, 128, 512, 152) == 0
    assert g(1, 1, 8, 2, 128, 512, 152) == lib.fa_decode_workspace_size(1, 8, 2, 128, 512, 152)
    assert g(2, 4, 8, 2, 128, 512, 152) >= g(2, 1, 8, 2, 128, 512, 152)


def test_batch_invariant_rejects_bad_split_and_sizes_its_workspace(lib):
    f = lib.fa_decode_batch_invariant
    #                q  k      v      vs    bt    sl     hq hkv d   scale win  out    B  P   maxb nblk
    args = lambda st: (A, 2 * A, 3 * A, None, None, 4 * A, 8, 2, 128, 0.1, None, 5 * A, 1, 16, 512, 0,
                       st, 6 * A, 1 << 30, None)
    for bad in (0, -16, 24, 8):
        assert f(*args(bad)) == -6, bad
        assert lib.fa_decode_last_error()
    g = lib.fa_decode_batch_invariant_workspace_size
    assert g(1, 8, 2, 128, 512, 0) == 0 and g(1, 8, 2, 128, 512, 8) == 0
    assert g(0, 8, 2, 128, 512, 512) == 0 and g(1, 6, 4, 128, 512, 512) == 0
    # one partial (D floats of O + max and sum) per query head of each unit
    # (2 KV heads x 4 heads) and split: 512 keys in 512-key splits is one
    one = g(1, 8, 2, 128, 512, 512)
    assert one == 2 * 1 * 4 * (128 * 4 + 8)
    assert g(1, 8, 2, 128, 512, 16) == 32 * one
    assert g(3, 8, 2, 128, 512, 512) == 3 * one
    assert g(1, 8, 2, 128, 513, 512) == 2 * one


def test_batch_invariant_workspace_size_does_not_wrap(lib):
    """The scratch grows with batch x units x splits; where that passes 2^64
    bytes the size is 0 (invalid) rather than the wrapped remainder."""
    g = lib.fa_decode_batch_invariant_workspace_size
    h = lib.fa_decode_multi_batch_invariant_workspace_size
    B, Hkv, G, D, L = 65535, 4096, 64, 256, 1 << 30
    # one split per unit: 8 units of 8 heads per KV head, D floats + (m, l) each
    assert g(B, Hkv * G, Hkv, D, L, L) == B * Hkv * 8 * 8 * (D * 4 + 8)
    assert g(B, Hkv * G, Hkv, D, L, 16) == 0             # 2^26 splits per unit: > 2^64 bytes
    assert h(B, 256, Hkv * G, Hkv, D, L, 16) == 0
    assert g(1, 8, 2, 128, L, 16) == 2 * (L // 16) * 4 * (128 * 4 + 8)


def test_batch_invariant_multi_and_ring_reject_bad_arguments(lib):
    f = lib.fa_decode_multi_batch_invariant
    #               q  k      v      vs    bt    sl     tq hq hkv d    scale win  out    B  P   maxb
    args = lambda tq, st: (A, 2 * A, 3 * A, None, None, 4 * A, tq, 8, 2, 128, 0.1, None, 5 * A, 1,
                           16, 512, 0, st, 6 * A, 1 << 30, None)
    assert f(*args(0, 512)) == -6 and f(*args(257, 512)) == -6
    assert f(*args(4, 24)) == -6 and f(*args(4, 0)) == -6
    g = lib.fa_decode_ring_batch_invariant
    #        q  k      v      vs    sl     hq hkv d    scale win  out    B  cap  st   ws     wsb
    assert g(A, 2 * A, 3 * A, None, 4 * A, 8, 2, 128, 0.1, None, 5 * A, 1, 100, 512, 6 * A,
             1 << 30, None) == -6
    assert g(A, 2 * A, 3 * A, None, 4 * A, 8, 2, 128, 0.1, None, 5 * A, 1, 64, 40, 6 * A,
             1 << 30, None) == -6
    h = lib.fa_decode_multi_batch_invariant_workspace_size
    assert h(1, 0, 8, 2, 128, 512, 512) == 0 and h(1, 4, 8, 2, 128, 512, 24) == 0
    # one query is the single-query plan; 4 queries x G=4 = 16 columns = two
    # 8-column units per KV head
    assert h(1, 1, 8, 2, 128, 512, 512) == lib.fa_decode_batch_invariant_workspace_size(
        1, 8, 2, 128, 512, 512)
    assert h(1, 4, 8, 2, 128, 512, 512) == 2 * 2 * 1 * 8 * (128 * 4 + 8)


def test_missing_library_fails_loudly(tmp_path):
    """No CPU or PyTorch fallback: without the built library (or with a build
    that fails) the first call raises instead of computing anything."""
    import subprocess
    import sys
    code = f"""
import torch
from decode_step_kv_gb300 import _build, binding
_build.LIB = {str(tmp_path / "absent.so")!r}
try:
    binding.load(build_if_missing=False)
except OSError:
    print("absent: raised")
def broken(*a, **k):
    raise RuntimeError("nvcc failed")
_build.build = broken
try:
    binding.fa_decode_workspace_size(1, 8, 2, 128, 512, 152)
except RuntimeError as e:
    print("build:", e)
"""
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert "absent: raised" in r.stdout and "build: nvcc failed" in r.stdout, r.stdout


def test_slots_reject_bad_arguments(lib):
    f = lib.fa_decode_slots
    #             q  k      v      vs    slots  sl     hq hkv d    scale win  out    B  n   cap  ring
    def args(**kw):
        a = dict(q=A, k=2 * A, v=3 * A, vs=None, si=7 * A, sl=4 * A, out=5 * A, ns=64, cap=512,
                 ring=0)
        a.update(kw)
        return (a["q"], a["k"], a["v"], a["vs"], a["si"], a["sl"], 8, 2, 128, 0.1, None,
                a["out"], 1, a["ns"], a["cap"], a["ring"], 6 * A, 1 << 30, None)
    assert f(*args(si=None)) == -1
    assert f(*args(ns=0)) == -6
    assert f(*args(cap=0)) == -6
    assert f(*args(ring=1, cap=100)) == -6               # a ring's capacity: a multiple of 16
    assert f(*args(vs=8 * A, cap=100)) == -6             # contiguous int8 V likewise
    assert f(*args(si=7 * A + 2)) == -9                  # slot_ids: 4-byte aligned
    assert f(*args(out=7 * A)) == -7                     # out over the slot map
    g = lib.fa_append_kv_slots
    #               k_new v_new k_cache v_cache sc  slots pos  B  Hkv D   n   cap ring
    def gargs(**kw):
        a = dict(si=7 * A, pos=4 * A, ns=8, cap=64, ring=0, kn=A)
        a.update(kw)
        return (a["kn"], A + 4096, 2 * A, 3 * A, None, a["si"], a["pos"], 1, 2, 128, a["ns"],
                a["cap"], a["ring"], None)
    assert g(*gargs(si=None)) == -1
    assert g(*gargs(ns=0)) == -6
    assert g(*gargs(ring=1, cap=40)) == -6
    assert g(*gargs(si=7 * A + 1)) == -9
    # the K pool (8 slots x 2 x 64 x 128 fp16 = 256 KiB from 2A) would hold the slot map
    assert g(*gargs(si=2 * A + 65536)) == -7
