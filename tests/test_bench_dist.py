"""The multi-rank path of bench.py on CPU: two gloo ranks launched the way
the benchmark is launched on several GPUs (torch.distributed.run, rendezvous
on 127.0.0.1)."""
import json
import os
import re
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    # the ranks share one pipe, so their lines may run together: take every object
    return [json.loads(m) for m in re.findall(r"\{(?:[^{}]|\{[^{}]*\})*\}", r.stdout)]


def test_slowest_rank_sets_the_job_time():
    lines = _torchrun([os.path.join("tests", "dist_worker.py")], timeout=120)
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["world"] == 2
        assert l["slowest_ms"] == 2.5                     # max over ranks of 1.5 and 2.5
        assert abs(l["value"] - 16800.0) < 1e-6          # both ranks' 21 alphas in the slowest 2.5 ms


def test_reference_arm_prints_one_line_from_rank_zero():
    lines = _torchrun(["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                       "--config", "tiny-128x256-n64"], timeout=300)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["value"] > 0
