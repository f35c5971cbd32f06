"""The N>1 host path of bench.py, on CPU: two ranks over gloo.

Each rank runs its own replica of the workload; the only exchange is the
whole-job reduction after the timed region (the slowest rank's time, the sum of
all ranks' tokens), and only rank 0 prints. The ranks are plain processes with
the environment torchrun would give them, rendezvous on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import io, json, sys, contextlib, argparse
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, world, local = bench.dist_env()
dist.init_process_group("gloo")
assert dist.get_rank() == rank and dist.get_world_size() == world
t_dev = [0.50, 0.75][rank]
tokens = [100, 140][rank]
t_all, tok_all = bench.over_ranks(t_dev, tokens, "cpu")
# the reference arm: every rank but 0 leaves at once, without output or work
buf = io.StringIO()
if rank != 0:
    with contextlib.redirect_stdout(buf):
        bench.run_reference(argparse.Namespace(steps=1, warmup=0, gpus=world))
dist.barrier()
dist.destroy_process_group()
print(json.dumps({{"rank": rank, "world": world, "local": local, "t": t_all, "tokens": tok_all,
                  "ref_out": buf.getvalue()}}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_gloo_reduction_and_rank0_only_reference():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, e[-2000:]
        outs.append(json.loads(o.strip().splitlines()[-1]))
    for r, d in enumerate(outs):
        assert (d["rank"], d["world"], d["local"]) == (r, 2, r)
        assert d["t"] == 0.75          # max over ranks
        assert d["tokens"] == 240.0    # sum over ranks
    assert outs[1]["ref_out"] == ""


def test_single_process_reduction_is_identity(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.over_ranks(0.25, 37, "cpu") == (0.25, 37.0)
