"""The multi-GPU plumbing of bench.py on CPU: `--gpus N` runs N independent replicas (the P
logical ranks of the method live on one GPU, so replicas exchange nothing on the data path).
Two gloo ranks check the barrier and the max-over-ranks reduction that the bench's timing uses,
and that a rank other than 0 prints nothing in the reference arm."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import bench
r = bench.Ranks(2)
r.barrier()
t = r.max(float(r.rank) + 0.5)
r.barrier()
print(json.dumps({"rank": r.rank, "world": r.world, "max": t}), flush=True)
r.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_two_ranks(code: str, extra_args=()):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code, ROOT, *extra_args], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            out, err = p.communicate()
        outs.append((p.returncode, out, err))
    return outs


def test_two_gloo_replicas_barrier_and_max():
    outs = _run_two_ranks(_CHILD)
    import json
    seen = []
    for rc, out, err in outs:
        assert rc == 0, err
        rec = json.loads(out.strip().splitlines()[-1])
        assert rec["world"] == 2
        assert rec["max"] == 1.5          # max over ranks of rank + 0.5
        seen.append(rec["rank"])
    assert sorted(seen) == [0, 1]


_REF_CHILD = r"""
import os, sys
sys.path.insert(0, sys.argv[1])
import bench, inputgen as ig

class Args:
    warmup, steps, gpus, reference_step_s = 0, 1, 2, 0.05
    split, tiles = "chained", "pair"

r = bench.Ranks(2)
wl = ig.WORKLOADS["ar_p2_m128_n128_k256"]
bench.reference_arm(Args, wl, r)
r.barrier()
r.close()
"""


def test_reference_arm_prints_only_on_rank_0():
    outs = _run_two_ranks(_REF_CHILD)
    lines = []
    for rc, out, err in outs:
        assert rc == 0, err
        lines.append([l for l in out.splitlines() if l.startswith("{")])
    assert sum(len(l) for l in lines) == 1    # one JSON line in all
