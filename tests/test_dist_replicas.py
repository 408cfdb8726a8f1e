"""The N-GPU bench path runs independent replicas (no collective on the data
path); its only cross-rank steps are the barrier around the timed region and
the max of the step time over ranks.  Both run here as two gloo ranks on CPU."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r'''
import os, sys
sys.path.insert(0, ROOT)
import torch.distributed as dist
import bench
world, rank, local = bench.dist_setup(None)
assert world == 2 and dist.get_backend() == "gloo"
bench.barrier(world)
m = bench.max_over_ranks(10.0 + rank, world)
print(f"rank{rank} max={m}", flush=True)
dist.destroy_process_group()
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code, nproc=2):
    port = _free_port()
    procs = []
    for r in range(nproc):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(nproc),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code.replace("ROOT", repr(ROOT))],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    return [(p.returncode, o, e) for p, (o, e) in zip(procs, outs)]


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    res = _launch(RANK_SCRIPT)
    for rc, out, err in res:
        assert rc == 0, err[-2000:]
    assert "rank0 max=11.0" in res[0][1]
    assert "rank1 max=11.0" in res[1][1]


def test_reference_arm_prints_on_rank_zero_only():
    code = r'''
import sys
sys.path.insert(0, ROOT)
sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
import bench
bench.oracle_sample = lambda wl, inp, budget_s, threads=0: (1.0, 0.01, 1, 1)
bench.cpu_inputs = lambda wl: {}
bench.main()
'''
    res = _launch(code)
    for rc, out, err in res:
        assert rc == 0, err[-2000:]
    assert '"impl": "reference"' in res[0][1]
    assert res[1][1].strip() == ""
