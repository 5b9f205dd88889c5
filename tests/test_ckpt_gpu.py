"""State checkpoints (kda_chunk_fwd_ckpt): the state after every `every`
tokens of each sequence equals the oracle's final state of that prefix."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_32_gb300 import kda
from kda_inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gated_delta_rule_32_gb300 import build
    build.build()
    kda.load()


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, 1e-2), (torch.float32, 1e-4)])
@pytest.mark.parametrize("varlen", [False, True])
def test_checkpoints(dtype, tol, varlen):
    every, maxc = 64, 4
    if varlen:
        lens = (100, 200, 70, 257)
        w = small_workload("ck", B=1, T=sum(lens), H=2, dk=128, dv=128, dtype=dtype, seed=4,
                           varlen=True, lengths=lens, s0_std=0.02)
    else:
        lens = (300, 300)
        w = small_workload("ck", B=2, T=300, H=2, dk=128, dv=128, dtype=dtype, seed=4,
                           s0_std=0.02)
    x = make_inputs(w)
    N, H = x["B"], w.H
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    out = torch.empty_like(d["v"])
    fs = torch.empty(N, H, 128, 128, device="cuda")
    ck = torch.full((N, H, maxc, 128, 128), float("nan"), device="cuda")
    dt = kda.KDA_BF16 if dtype == torch.bfloat16 else kda.KDA_F32
    rc = kda.kda_chunk_fwd_ckpt(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], out,
                                fs, N, x["T"], H, 128, 128, d["cu_seqlens"], dt, 1.0, ck, every,
                                maxc, None, torch.cuda.current_stream())
    assert rc == 0
    torch.cuda.synchronize()
    ck = ck.cpu().numpy()
    starts = np.concatenate([[0], np.cumsum(lens)])
    for n in range(N):
        L = lens[n]
        for c in range(maxc):
            t_end = (c + 1) * every
            if t_end > L:
                assert np.isnan(ck[n, :, c]).all()      # slot never written
                continue
            if varlen:
                sl = slice(starts[n], starts[n] + t_end)
                args = [x[key][:, sl] for key in ("q", "k", "v", "g", "beta")]
            else:
                args = [x[key][n:n + 1, :t_end] for key in ("q", "k", "v", "g", "beta")]
            _, s_ref = oracle.fwd(*args, x["init_state"][n:n + 1])
            assert rel(ck[n, :, c], s_ref[0]) <= tol, (n, c)


def test_checkpoint_arguments():
    A = 1 << 20
    bad = dict(checkpoints=7 * A, every=100, max_per_seq=2)
    rc = kda.kda_chunk_fwd_ckpt(A, 2 * A, 3 * A, 4 * A, 5 * A, None, 6 * A, None, 1, 64, 1, 128,
                                128, None, kda.KDA_BF16, 1.0, **bad)
    assert rc == kda.KDA_ERR_INVALID_ARG
