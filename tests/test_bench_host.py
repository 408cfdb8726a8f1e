"""Host-side checks of the benchmark's bookkeeping (no GPU needed).

bench.py reports `roofline.traffic` from the committed ncu summary only while
that summary was taken on the kernel source being timed.
"""
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join("decode_step_kv_gb300", "csrc", "fa_decode.cu")
SUMMARY = os.path.join("profiles", "fa_stream_mma_kernel_4x1k-8k_d256.md")


def _tree(tmp_path, source_text):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "decode_step_kv_gb300" / "csrc").mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, SUMMARY), tmp_path / SUMMARY)
    (tmp_path / SRC).write_bytes(source_text)


def test_traffic_is_read_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    real = open(os.path.join(ROOT, SRC), "rb").read()
    committed = bench.recorded_traffic("fa_stream_mma_kernel", "4x1k-8k_d256")
    assert committed is not None and committed > 0      # the committed summary matches the tree
    _tree(tmp_path, real)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("fa_stream_mma_kernel", "4x1k-8k_d256") == committed
    (tmp_path / SRC).write_bytes(real + b"\n")        # any change to the kernel source
    assert bench.recorded_traffic("fa_stream_mma_kernel", "4x1k-8k_d256") is None
    assert bench.recorded_traffic("fa_stream_mma_kernel", "no_such_workload") is None

