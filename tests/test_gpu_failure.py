"""Failure detection on the GPU without a fault: a wait that can never be
satisfied gives up after its ~1 s bound, reports FA_STATUS_WAIT_TIMEOUT, and
the context keeps working for the next decode call."""
import time

import pytest
import torch

from decode_step_kv_gb300 import binding
from decode_step_kv_gb300.inputs import Workload

from _helpers import assert_close, build_case, gpu_decode, oracle_decode, to_cuda

pytestmark = pytest.mark.gpu


def test_unsatisfiable_wait_times_out_and_reports():
    binding.fa_decode_device_status()                         # clear earlier bits
    t0 = time.perf_counter()
    binding.fa_selftest_wait_timeout()
    status = binding.fa_decode_device_status()                # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status & binding.FA_STATUS_WAIT_TIMEOUT
    assert 0.5 < elapsed < 30.0
    # the context is still usable
    wl = Workload("after_timeout", 2, 8, 2, 128, paged=True, seed=3)
    inp = build_case(wl, seq_lens=[100, 700])
    got = gpu_decode(wl, to_cuda(inp)).cpu().numpy()
    assert_close(got, oracle_decode(wl, inp), False, "after timeout")
    assert binding.fa_decode_device_status() == 0
