"""The oracle's pins catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of oracle/fa_oracle.c: a dropped
term, an off-by-one bound, a wrong index, a swapped operand or a different
rounding rule.  The copy is compiled like the oracle, swapped in for it, and
the pin tests (closed forms, brute force, golden values, equivalences) are run
against it: at least one must fail.  The unchanged source, compiled the same
way, passes them all, so a failure comes from the planted mistake and not from
the harness.  Every planted variant stays inside the arrays it is given.
"""
import ctypes
import importlib
import itertools
import os
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fa_oracle.c")
PIN_MODULES = ["test_oracle_pins", "test_oracle_multi", "test_oracle_ring", "test_oracle_append",
               "test_oracle_slots"]

# (name, text in fa_oracle.c, replacement); the text must occur in the file
MUTANTS = [
    ("scale dropped",
     "double s = P->scale * dot;", "double s = dot;"),
    ("last head_dim term dropped",
     "for (int d = 0; d < P->D; ++d)\n            dot +=",
     "for (int d = 0; d < P->D - 1; ++d)\n            dot +="),
    ("query head mapped to kv head h % Hkv",
     "int kv = h / (P->Hq / P->Hkv);", "int kv = h % P->Hkv;"),
    ("window one key short",
     "*lo = (W > 0 && end > W) ? end - W : 0;", "*lo = (W > 0 && end > W) ? end - W + 1 : 0;"),
    ("window one key long",
     "*lo = (W > 0 && end > W) ? end - W : 0;", "*lo = (W > 0 && end > W) ? end - W - 1 : 0;"),
    ("softmax not normalised",
     "p[t - lo] /= z;", "p[t - lo] /= 1.0;"),
    ("softmax sign flipped",
     "p[t - lo] = exp(p[t - lo] - smax);", "p[t - lo] = exp(smax - p[t - lo]);"),
    ("base-2 exponent without the log2(e) factor",
     "p[t - lo] = exp(p[t - lo] - smax);", "p[t - lo] = exp2(p[t - lo] - smax);"),
    ("keys read from the range start instead of their position",
     "const uint16_t *krow = P->k + row_offset(P, b, kv, t, P->D);",
     "const uint16_t *krow = P->k + row_offset(P, b, kv, t - lo, P->D);"),
    ("int8 scale of the wrong 32-block",
     "row_offset(P, b, kv, t, P->D / 32) + d / 32]",
     "row_offset(P, b, kv, t, P->D / 32) + d % (P->D / 32)]"),
    ("int8 scale amax / 128",
     "oracle_double_to_half(amax / 127.0)", "oracle_double_to_half(amax / 128.0)"),
    ("int8 codes truncated",
     "qv = rint((double)xb[i] / s);", "qv = trunc((double)xb[i] / s);"),
    ("fp16 encode truncates",
     "double r = rint(ax / ulp) * ulp;", "double r = floor(ax / ulp) * ulp;"),
    ("row within a page shifted",
     "int r = t % P->page_size;", "int r = (t + 1) % P->page_size;"),
    ("ring row shifted",
     "long long r = P->ring ? t % P->max_blocks : t;",
     "long long r = P->ring ? (t + 1) % P->max_blocks : t;"),
    ("ring keeps one token too few",
     "*lo = *hi - P->max_blocks;", "*lo = *hi - P->max_blocks + 1;"),
    ("query j cut one key early",
     "int end = L - (tq - 1 - j);", "int end = L - (tq - j);"),
    ("append K row takes the V values",
     "k_cache[row * D + d] = oracle_double_to_half((double)kr[d]);",
     "k_cache[row * D + d] = oracle_double_to_half((double)vr[d]);"),
    ("append to the next contiguous row",
     "row = (slot * Hkv + kv) * max_blocks + t;",
     "row = (slot * Hkv + kv) * max_blocks + (t + 1) % max_blocks;"),
    ("slot map ignored: row b reads slot b",
     "return ((slot_of(P, b) * P->Hkv + kv) * P->max_blocks + r) * (long long)row_elems;",
     "return (((long long)b * P->Hkv + kv) * P->max_blocks + r) * (long long)row_elems;"),
    ("append through the slot map writes slot b",
     "            slot = slot_ids[b];\n", "            slot = b;\n"),
    ("gather reads the row after",
     "off = ((blk * Hkv + kv) * page_size + t % page_size) * (long long)row_bytes;",
     "off = ((blk * Hkv + kv) * page_size + (t + 1) % page_size) * (long long)row_bytes;"),
]


def _compile(text, path):
    with open(path + ".c", "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-w", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", path, path + ".c", "-lm", "-lpthread"], check=True)
    return oracle._configure(ctypes.CDLL(path))


def _pin_calls():
    """Every pin test of the oracle modules, with each parametrisation."""
    calls = []
    for name in PIN_MODULES:
        mod = importlib.import_module(name)
        for attr in sorted(dir(mod)):
            fn = getattr(mod, attr)
            if not (attr.startswith("test_") and callable(fn)):
                continue
            grids = []
            for mark in getattr(fn, "pytestmark", []):
                if mark.name == "parametrize":
                    names = [n.strip() for n in mark.args[0].split(",")]
                    values = [v if len(names) > 1 else (v,) for v in mark.args[1]]
                    grids.append([dict(zip(names, v)) for v in values])
            for combo in itertools.product(*grids):
                kw = {}
                for part in combo:
                    kw.update(part)
                calls.append((f"{name}.{attr}", fn, kw))
    return calls


def _failures(lib):
    """The pin calls that fail with `lib` standing in for the oracle."""
    saved = oracle._lib
    oracle._lib = lib
    failed = []
    try:
        for label, fn, kw in _pin_calls():
            try:
                fn(**kw)
            except Exception as e:                  # an assertion or a rejected call
                failed.append(f"{label}{kw or ''}: {type(e).__name__}")
    finally:
        oracle._lib = saved
    return failed


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


def test_unchanged_source_passes_every_pin(source, tmp_path):
    lib = _compile(source, str(tmp_path / "same.so"))
    assert _failures(lib) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(source, tmp_path, name, old, new):
    assert old in source, f"mutation site of {name!r} not found"
    lib = _compile(source.replace(old, new), str(tmp_path / "mutant.so"))
    failed = _failures(lib)
    assert failed, f"no pin catches: {name}"
