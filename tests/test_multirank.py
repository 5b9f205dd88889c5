"""The multi-GPU path of bench.py on CPU: two ranks under torchrun with the
gloo backend (rendezvous on 127.0.0.1).  Each rank runs an independent batch
(its own seed), there is no collective on the data path, the time is the
slowest rank's and the value counts every rank's tokens (weak scaling); the
reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=300):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, OMP_NUM_THREADS="1")
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout,
                          env=env)


def test_two_ranks_weak_scaling_pieces():
    r = _torchrun([os.path.join("tests", "_multirank_worker.py")])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    by = {d["rank"]: d for d in lines}
    assert by[0]["ws"] == by[1]["ws"] == 2
    assert by[0]["seed"] != by[1]["seed"]          # independent batches
    assert by[0]["q0"] != by[1]["q0"]
    for d in lines:                                 # the slowest rank's time
        assert d["slowest_ms"] == 15.0
        assert abs(d["value"] - 2 * 2 * 32768 / 0.015) < 1e-3 * d["value"]


def test_reference_arm_on_rank_zero_only():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "1", "--ref-units", "1", "--ref-tokens", "128"])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                           # one JSON line, from rank 0
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["scaling"] == "weak" and d["cpu_baseline"]["kind"] == "oracle"
