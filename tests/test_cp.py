"""Context parallelism across ranks on the CPU: the exchange and the scan.

World sizes 2 and 3 over gloo on 127.0.0.1, uneven token spans.  Each rank
runs gated_delta_rule_32_gb300.cp.context_parallel_forward with the three
per-rank steps taken from the fp64 oracle (span summary, composition of the
gathered summaries, the span's forward from the composed entry state).  The
concatenated outputs must equal the oracle's forward of the whole batch, and
rank r's state after its span must equal the oracle's state after tokens
[0, t_{r+1}): a wrong order of the gathered summaries, a missing or extra
fold, or a transposed composition fails.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
from kda_inputs import make_inputs, small_workload
from tests import _cp_worker


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run_ranks(world, mode, tmp_path, B, T, H, d, seed):
    mp.spawn(_cp_worker.run, args=(world, _free_port(), mode, str(tmp_path), B, T, H, d, seed),
             nprocs=world, join=True)
    return [dict(np.load(os.path.join(tmp_path, "rank%d.npz" % r))) for r in range(world)]


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_exchange_and_scan(world, tmp_path):
    B, T, H, d, seed = 2, 90, 2, 8, 33
    ranks = run_ranks(world, "oracle", tmp_path, B, T, H, d, seed)
    w = small_workload("cp", B=B, T=T, H=H, dk=d, dv=d, seed=seed, s0_std=0.05,
                       dtype=__import__("torch").float32)
    x = make_inputs(w)
    o_ref, s_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["init_state"])
    out = np.concatenate([r["out"] for r in ranks], axis=1)
    den = np.abs(o_ref).max()
    assert np.abs(out - o_ref).max() <= 1e-10 * den
    for r in ranks:
        t1 = int(r["t1"])
        _, s_t1 = oracle.fwd(x["q"][:, :t1], x["k"][:, :t1], x["v"][:, :t1], x["g"][:, :t1],
                             x["beta"][:, :t1], x["init_state"])
        assert np.abs(r["state"] - s_t1).max() <= 1e-10 * np.abs(s_t1).max()
    np.testing.assert_allclose(ranks[-1]["state"], s_ref, rtol=0, atol=1e-10 * np.abs(s_ref).max())
