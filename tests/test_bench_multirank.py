"""The bench's multi-rank host logic on CPU (gloo, world size 2): the timed
region is the slowest rank's, the value is the whole job's (weak scaling),
and under torchrun the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as tdist
import bench
rank = int(os.environ["RANK"])
tdist.init_process_group("gloo", init_method="env://")
# rank 0 was slower in the first value, rank 1 in the second
local = [10.0 if rank == 0 else 7.5, 3.0 if rank == 0 else 4.25]
red = bench.max_over_ranks(local, "cpu")
rate = bench.whole_job_rate(1000.0, 5, tdist.get_world_size(), red[0])
tdist.barrier()
tdist.destroy_process_group()
with open(os.path.join({out!r}, f"r{{rank}}.json"), "w") as f:
    json.dump({{"red": red, "rate": rate}}, f)
"""


def _run_two(code_fn, tmp_path, extra_env=None):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   LOCAL_RANK=str(rank), WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code_fn(rank)], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=120)
        outs.append((p.returncode, o, e))
    return outs


def test_max_over_ranks_and_whole_job_rate(tmp_path):
    outs = _run_two(lambda r: WORKER.format(root=ROOT, out=str(tmp_path)), tmp_path)
    for rc, o, e in outs:
        assert rc == 0, e[-2000:]
    import json
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["red"] == [10.0, 4.25]                  # the slowest rank, per entry
        assert r["rate"] == pytest.approx(2 * 1000.0 * 5 / 0.010)   # both ranks' work / max time


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    # rank 1 of a reference run exits 0 at once and prints nothing; rank 0's
    # run is the oracle (too slow for this test), so only rank 1 is started
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()), CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
