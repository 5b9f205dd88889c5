"""Child process of tests/test_threads_gpu.py: the first calls of a fresh
process into libkda.so come from two host threads at once, each on its own
stream; then the same calls run one after the other.  Prints one JSON line
saying whether every concurrent result equals its serial twin bit for bit.
"""
import json
import os
import sys
import threading

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_delta_rule_32_gb300 import kda  # noqa: E402
from kda_inputs import make_inputs, small_workload  # noqa: E402


def main():
    kda.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # two shapes on two different paths (the two-kernel path and the fused
    # kernel), so each thread's first call sets up different kernels
    jobs = []
    for i, algo in enumerate((kda.KDA_ALGO_AUTO, kda.KDA_ALGO_TC)):
        w = small_workload("thr%d" % i, B=2, T=300 + 70 * i, H=3, seed=40 + i, s0_std=0.05)
        x = make_inputs(w)
        d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
        jobs.append((w, d, algo))
    torch.cuda.synchronize()

    def run(j, stream, res, slot):
        w, d, algo = jobs[j]
        out = torch.full_like(d["v"], float("nan"))
        fs = torch.full((w.B, w.H, 128, 128), float("nan"), device=dev)
        with torch.cuda.stream(stream):
            rc = kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                      d["init_state"], out, fs, w.B, w.T, w.H, 128, 128, None,
                                      kda.KDA_BF16, 0, 1.0, algo, None, 0, None, stream)
        stream.synchronize()
        res[slot] = (rc, out, fs)

    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    conc = [None, None]
    barrier = threading.Barrier(2)

    def worker(j):
        barrier.wait()
        run(j, streams[j], conc, j)
    ts = [threading.Thread(target=worker, args=(j,)) for j in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    ser = [None, None]
    for j in range(2):
        run(j, streams[0], ser, j)
    ok = all(conc[j][0] == 0 and ser[j][0] == 0 and torch.equal(conc[j][1], ser[j][1]) and
             torch.equal(conc[j][2], ser[j][2]) for j in range(2))
    print(json.dumps({"ok": bool(ok), "rc": [conc[0][0], conc[1][0], ser[0][0], ser[1][0]]}))


if __name__ == "__main__":
    main()
