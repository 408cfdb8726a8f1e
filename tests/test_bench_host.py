"""Host-side checks of the benchmark's bookkeeping (no GPU needed).

bench.py reports `roofline.traffic` from the committed ncu summary only while
that summary was taken on the kernel source being timed.
"""
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join("decode_step_kv_gb300", "csrc", "fa_decode.cu")


def _tree(tmp_path, source_text, summary_text):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "decode_step_kv_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "profiles" / "fa_stream_mma_kernel_w.md").write_text(summary_text)
    (tmp_path / SRC).write_bytes(source_text)


def test_traffic_is_read_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    import hashlib
    real = open(os.path.join(ROOT, SRC), "rb").read()
    summary = (f"Kernel source: x, source sha256: {hashlib.sha256(real).hexdigest()}\n"
               "- traffic_bytes_per_launch: 4295000000 (scaled)\n")
    _tree(tmp_path, real, summary)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("fa_stream_mma_kernel", "w") == 4295000000
    (tmp_path / SRC).write_bytes(real + b"\n")        # any change to the kernel source
    assert bench.recorded_traffic("fa_stream_mma_kernel", "w") is None
    assert bench.recorded_traffic("fa_stream_mma_kernel", "no_such_workload") is None


def test_e2e_copies_send_written_rows_of_a_contiguous_cache():
    """The end-to-end leg sends each (sequence, KV head)'s rows [0, L_b) of a
    contiguous cache, at the same place on both sides, and everything else
    whole; a paged pool goes whole."""
    import dataclasses

    import torch

    from decode_step_kv_gb300.inputs import Workload
    wl = Workload("t", 3, 4, 2, 128)
    lens = [5, 0, 16]
    cap = 16
    host = {"q": torch.randn(3, 4, 128).half(),
            "k_cache": torch.randn(3, 2, cap, 128).half(),
            "v_cache": torch.randint(-127, 128, (3, 2, cap, 128), dtype=torch.int8),
            "v_scales": torch.randn(3, 2, cap, 4).half(),
            "seq_lens": torch.tensor(lens, dtype=torch.int32)}
    dev = {n: torch.zeros_like(t) for n, t in host.items()}
    copies = bench.e2e_copies(wl, lens, host, dev)
    row = 128 * 2 + 128 + 4 * 2                  # K fp16 + V int8 + scales, per token
    assert sum(s.numel() * s.element_size() for _, s in copies) == \
        sum(lens) * 2 * row + 3 * 4 * 128 * 2 + 3 * 4
    for dst, src in copies:
        assert src.is_contiguous() and dst.is_contiguous()
        dst.copy_(src)
    for n in ("k_cache", "v_cache", "v_scales"):
        for b, L in enumerate(lens):
            assert torch.equal(dev[n][b, :, :L], host[n][b, :, :L])
            assert not dev[n][b, :, L:].any()     # padding rows were not sent
    paged = dataclasses.replace(wl, paged=True)
    pool = {"k_cache": torch.randn(7, 2, 16, 128).half()}
    assert [(d.shape, s.shape) for d, s in bench.e2e_copies(paged, lens, pool,
                                                             {"k_cache": pool["k_cache"]})] == \
        [(pool["k_cache"].shape, pool["k_cache"].shape)]


def test_clock_summary_reads_median_max_and_active_reasons():
    """nvidia-smi csv,noheader,nounits lines -> median SM clock, max clock
    and the throttle reasons seen Active; malformed lines are skipped."""
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 900.10, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1100.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
        "0, [N/A], 2070, 1.0, 0x0, Active, Active, Active, Active",
    ]
    got = s.summary()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}
    s.lines = ["0, 1500, 2070, 500.0, 0x8, Not Active, Active, Not Active, Not Active"]
    assert s.summary()["reasons"] == ["hw_thermal_slowdown"]
    s.lines = []
    assert s.summary() is None
